"""GPU parity of the output-copy cross-attention (Eq. 5) with many copies per
sequence (T_out * G >= 256: the tensor-memory flash kernel) against the fp64
oracle: SFT answer spans, PT mode (a copy at every position), partial last
tiles, rows of very different lengths in one CTA, duplicates, and rejected
positions (zero rows, ORTHROS_DEVERR_POSITION)."""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import PrefillConfig, make_prefill
from tests.gpu_util import assert_parity, bf, dev, f32, i32, val

pytestmark = pytest.mark.gpu


def _xattn(inp, pos=None):
    cfg = inp.cfg
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    p = inp.pos if pos is None else pos
    qc = bf(inp.q_raw)[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    oc = orth.xattn_fwd(qc, i32(p), bf(inp.k), bf(inp.v), f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale,
                        dev_err=err)
    torch.cuda.synchronize()
    return val(oc), int(err.item())


def _ref(inp, pos, sel=None):
    q = inp.qc_raw if sel is None else inp.qc_raw[:, sel]
    ps = pos if sel is None else pos[:, sel]
    return oracle.xattn(np.ascontiguousarray(q), np.ascontiguousarray(ps), inp.k, inp.v, inp.alpha_c, inp.beta_c,
                        inp.cfg.scale)


@pytest.mark.parametrize("B,T,Hq,Hkv,d,T_out", [
    (2, 1500, 32, 8, 128, 64),    # 256 rows per KV head: one full tile pair
    (1, 2000, 32, 8, 128, 100),   # a partial second tile pair
    (1, 900, 8, 4, 64, 160),      # G=2, d=64
    (1, 700, 16, 2, 128, 40),     # G=8
    (1, 600, 16, 1, 64, 20),      # G=16
])
def test_many_copies_parity(B, T, Hq, Hkv, d, T_out):
    cfg = PrefillConfig("many", B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, T_out=T_out)
    inp = make_prefill(cfg, 3000 + T_out)
    g = np.random.default_rng(T_out)
    # any positions: block edges, the ends, duplicates
    pos = g.integers(0, T, size=(B, T_out)).astype(np.int32)
    pos[:, :6] = [0, 127, 128, 255, T - 1, T - 1]
    got, err = _xattn(inp, pos)
    assert err == 0
    assert_parity(got, _ref(inp, pos), "many copies")


def test_pt_mode_every_position():
    """PT mode: one copy per position, physically shuffled."""
    cfg = PrefillConfig("pt", B=1, T=1024, Hq=8, Hkv=2, d=128, T_out=1024, positions="shuffled")
    inp = make_prefill(cfg, 61)
    got, err = _xattn(inp)
    assert err == 0
    assert_parity(got, _ref(inp, inp.pos), "PT copies")


def test_sft_appended_many_copies():
    cfg = PrefillConfig("sft_many", B=2, T=3000, Hq=32, Hkv=8, d=128, T_out=300, appended=True,
                        positions="shuffled", needle_frac=0.002)
    inp = make_prefill(cfg, 62)
    got, err = _xattn(inp)
    assert err == 0
    assert_parity(got, _ref(inp, inp.pos), "SFT copies with scaled key rows")


def test_many_copies_rejected_positions():
    cfg = PrefillConfig("many_bad", B=1, T=800, Hq=32, Hkv=8, d=128, T_out=80)
    inp = make_prefill(cfg, 63)
    pos = np.random.default_rng(5).integers(0, 800, size=(1, 80)).astype(np.int32)
    pos[0, [3, 40, 79]] = [-1, 800, 5000]
    got, err = _xattn(inp, pos)
    assert err & orth.DEVERR_POSITION
    assert (got[0, [3, 40, 79]] == 0).all()
    ok = np.setdiff1d(np.arange(80), [3, 40, 79])
    assert_parity(got[:, ok], _ref(inp, pos, ok), "valid copies next to rejected ones")


def test_many_copies_all_rejected():
    """No valid position in a whole CTA: zero rows, no key block streamed."""
    cfg = PrefillConfig("many_none", B=1, T=300, Hq=8, Hkv=2, d=128, T_out=64)
    inp = make_prefill(cfg, 64)
    pos = np.full((1, 64), -3, np.int32)
    got, err = _xattn(inp, pos)
    assert err & orth.DEVERR_POSITION
    assert (got == 0).all()


@pytest.mark.parametrize("boost_block", [1, 3])
def test_running_max_raised_in_the_second_half_of_a_key_pair(boost_block):
    """The tensor-memory kernel takes 128 keys per softmax step as two 64-key halves with a
    lazily raised running max.  Key block `boost_block` (the second half of a pair) scaled by
    4 (exact in bf16) makes its logits several times larger, so most rows raise their max there
    and the first half's already written weights must be rescaled in place; without that they
    would outweigh the second half by about 2^9."""
    from synthetic import bf16_bits, bf16_to_f32
    cfg = PrefillConfig("raise", B=1, T=600, Hq=8, Hkv=2, d=128, T_out=64)
    inp = make_prefill(cfg, 4242 + boost_block)
    k = bf16_to_f32(inp.k)
    k[:, 64 * boost_block:64 * boost_block + 64] *= np.float32(4.0)
    inp.k[...] = bf16_bits(k)
    pos = np.full((cfg.B, cfg.T_out), cfg.T - 1, np.int32)
    pos[:, :8] = [64 * boost_block + 63, 64 * boost_block, 64 * boost_block - 1, 64 * boost_block + 64, 599, 300,
                  200, 127]
    got, err = _xattn(inp, pos)
    assert err == 0
    assert_parity(got, _ref(inp, pos), "running max raised in a pair's second half")
