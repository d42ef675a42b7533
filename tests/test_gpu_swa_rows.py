"""GPU checks of orthros_swa_fwd_rows (chunked prefill): chunks computed one call at a
time give the rows of one full orthros_swa_fwd call bit for bit, on the tensor-memory
kernel and on the streaming kernel for wide windows; a call writes no row outside its
range; misaligned ranges are rejected."""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
from synthetic import PrefillConfig, make_prefill
from tests.gpu_util import bf, dev, f32

pytestmark = pytest.mark.gpu

SENTINEL = -12345  # int16 bit pattern no kernel writes here


def _inputs(B, T, Hq, Hkv, d, w, seed):
    cfg = PrefillConfig("rows", B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, window=w)
    inp = make_prefill(cfg, seed)
    return cfg, bf(inp.q_raw), bf(inp.k), bf(inp.v), f32(inp.alpha), f32(inp.beta)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,w,cuts", [
    (2, 1000, 32, 8, 128, 128, [0, 256, 384, 1000]),    # tensor-memory kernel, ragged last chunk
    (1, 777, 8, 4, 64, 128, [0, 128, 640, 777]),         # G=2, d=64
    (1, 900, 8, 2, 128, 600, [0, 512, 900]),             # band too wide: streaming kernel
    (1, 640, 16, 1, 64, 128, [0, 128, 256, 384, 512, 640]),  # G=16
])
def test_chunks_equal_full_call(B, T, Hq, Hkv, d, w, cuts):
    cfg, q, k, v, a, b = _inputs(B, T, Hq, Hkv, d, w, 7000 + T)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    full = orth.swa_fwd(q, k, v, a, b, window=w, scale=cfg.scale, dev_err=err)
    out = torch.full((B, T, Hq, d), SENTINEL, dtype=torch.int16, device=dev()).view(torch.bfloat16)
    for r0, r1 in zip(cuts[:-1], cuts[1:]):
        orth.swa_fwd_rows(q, k, v, a, b, r0, r1, window=w, scale=cfg.scale, out=out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int16), full.view(torch.int16))


def test_one_chunk_writes_only_its_rows():
    cfg, q, k, v, a, b = _inputs(2, 700, 32, 8, 128, 128, 7100)
    out = torch.full((2, 700, 32, 128), SENTINEL, dtype=torch.int16, device=dev()).view(torch.bfloat16)
    full = orth.swa_fwd(q, k, v, a, b, window=128, scale=cfg.scale)
    orth.swa_fwd_rows(q, k, v, a, b, 256, 512, window=128, scale=cfg.scale, out=out)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy()
    assert (got[:, :256] == SENTINEL).all() and (got[:, 512:] == SENTINEL).all()
    assert np.array_equal(got[:, 256:512], full.view(torch.int16).cpu().numpy()[:, 256:512])


@pytest.mark.parametrize("r0,r1", [(64, 256), (0, 200), (256, 128), (-128, 0), (0, 1024)])
def test_bad_ranges_are_rejected(r0, r1):
    cfg, q, k, v, a, b = _inputs(1, 700, 8, 2, 128, 128, 7200)
    with pytest.raises(orth.OrthrosError):
        orth.swa_fwd_rows(q, k, v, a, b, r0, r1, window=128, scale=cfg.scale)
