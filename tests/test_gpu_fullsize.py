"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times (one orthros_prefill_fwd call per prefill), against the fp64 oracle:

* the 8B-class 128K prefill (B=2): every base output row and both copies;
* the 1M-token prefill with scaled key rows: 16384 seeded random base rows, the
  first window and the tail, the rows around every scaled key row, and the copy;
* the SFT layer (B=4, 2048 appended shuffled copies per sequence): every base row
  and every copy;
* 128 decode steps after a 131072-token cache: sampled steps, and the cache bit
  for bit after all of them.
"""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import CONFIGS, SEEDS, bf16_to_f32, make_decode, make_prefill
from tests.gpu_util import ParityAccumulator, assert_parity, bf, bits, dev, f32, i32, val

pytestmark = pytest.mark.gpu

CHUNK_ROWS = 8192  # oracle rows per call when every row is compared


def _run_prefill(cfg, inp):
    """One orthros_prefill_fwd call, as bench.py times it (for few copies the copies' pass runs
    beside the SWA kernel on a second stream); its outputs must also have orthros_swa_fwd's and
    orthros_xattn_fwd's bits."""
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q_all = bf(inp.q_raw)
    k, v = bf(inp.k), bf(inp.v)
    qc = q_all[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    o, oc = orth.prefill_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), qc, i32(inp.pos), f32(inp.alpha_c),
                             f32(inp.beta_c), window=cfg.window, scale=cfg.scale, dev_err=err)
    o_swa = orth.swa_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), window=cfg.window, scale=cfg.scale,
                         dev_err=err)
    oc_x = orth.xattn_fwd(qc, i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale,
                          dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(o.view(torch.int16), o_swa.view(torch.int16)), "prefill_fwd base output"
    assert torch.equal(oc.view(torch.int16), oc_x.view(torch.int16)), "prefill_fwd copy output"
    del q_all, k, v, qc, o_swa, oc_x
    return o, oc


def _compare_rows(inp, o_bits, bi, ti, acc):
    """Oracle rows (b, t) against the GPU's output bits o_bits [B, T, Hq, d], in chunks."""
    cfg = inp.cfg
    q = np.ascontiguousarray(inp.q_base)  # once: the SFT layout keeps copies after the base rows
    for c0 in range(0, bi.size, CHUNK_ROWS):
        b, t = bi[c0:c0 + CHUNK_ROWS], ti[c0:c0 + CHUNK_ROWS]
        ref = oracle.swa_rows(q, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale, b, t)
        acc.add(bf16_to_f32(o_bits[b, t]).astype(np.float64), ref)


def _compare_copies(inp, oc_bits, sel, acc, per_call=256):
    cfg = inp.cfg
    for c0 in range(0, sel.size, per_call):
        s = sel[c0:c0 + per_call]
        ref = oracle.xattn(np.ascontiguousarray(inp.qc_raw[:, s]), np.ascontiguousarray(inp.pos[:, s]),
                           inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
        acc.add(bf16_to_f32(oc_bits[:, s]).astype(np.float64), ref)


def _every_row(cfg):
    t = np.tile(np.arange(cfg.T, dtype=np.int32), cfg.B)
    b = np.repeat(np.arange(cfg.B, dtype=np.int32), cfg.T)
    return b, t


def test_prefill_128k_every_row():
    cfg = CONFIGS["prefill_128k"]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    o, oc = _run_prefill(cfg, inp)
    o_bits, oc_bits = bits(o), bits(oc)
    del o, oc
    acc = ParityAccumulator("prefill_128k every base row")
    _compare_rows(inp, o_bits, *_every_row(cfg), acc)
    acc.check()
    accc = ParityAccumulator("prefill_128k copies")
    _compare_copies(inp, oc_bits, np.arange(cfg.T_out), accc)
    accc.check()


def test_prefill_1m_sampled_rows_and_every_scaled_key():
    cfg = CONFIGS["prefill_1m"]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    o, oc = _run_prefill(cfg, inp)
    o_bits, oc_bits = bits(o), bits(oc)
    del o, oc
    g = np.random.default_rng(1)
    rand = g.integers(0, cfg.T, size=16384)
    edges = np.concatenate([np.arange(0, 200), np.arange(cfg.T - 64, cfg.T)])
    # rows whose window holds a scaled key row: the needle's own row, the next, the middle of
    # its window and the last row that still sees it
    near = (inp.needles[:, None] + np.array([0, 1, 64, cfg.window - 1])[None, :]).reshape(-1)
    near = near[near < cfg.T]
    ti = np.concatenate([rand, edges, near]).astype(np.int32)
    bi = np.zeros_like(ti)
    acc = ParityAccumulator("prefill_1m base rows")
    _compare_rows(inp, o_bits, bi, ti, acc)
    acc.check()
    assert acc.n >= (16384 + 4 * len(inp.needles) - 8) * cfg.Hq * cfg.d
    accc = ParityAccumulator("prefill_1m copy")
    _compare_copies(inp, oc_bits, np.arange(cfg.T_out), accc)
    accc.check()


def test_sft_16k_every_row_and_copy():
    cfg = CONFIGS["sft_16k"]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    o, oc = _run_prefill(cfg, inp)
    o_bits, oc_bits = bits(o), bits(oc)
    del o, oc
    acc = ParityAccumulator("sft_16k every base row")
    _compare_rows(inp, o_bits, *_every_row(cfg), acc)
    acc.check()
    accc = ParityAccumulator("sft_16k every copy")
    _compare_copies(inp, oc_bits, np.arange(cfg.T_out), accc)
    accc.check()


def test_decode_128k_full_size_sampled_steps():
    cfg = CONFIGS["decode_128k"]
    inp = make_decode(cfg, SEEDS[cfg.name])
    kc, vc = bf(inp.k_cache), bf(inp.v_cache)
    cl = i32(inp.cache_len)
    a, b, ac, bc = (f32(x) for x in (inp.alpha, inp.beta, inp.alpha_c, inp.beta_c))
    ws = orth._binding.decode_workspace(cfg.B, cfg.L_max, cfg.Hq, cfg.Hkv, cfg.d, dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    check = {0, 1, 63, 127}
    outs = {}
    for i in range(cfg.steps):
        o, oc = orth.decode_step(bf(inp.q_new[i]), bf(inp.qc_new[i]), bf(inp.k_new[i]), bf(inp.v_new[i]),
                                 kc, vc, cl, a, b, ac, bc, window=cfg.window, scale=cfg.scale,
                                 workspace=ws, dev_err=err)
        if i in check:
            outs[i] = (val(o), val(oc))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the cache after 128 steps: the initial rows plus the appended ones, bit for bit
    expect_k, expect_v = inp.k_cache.copy(), inp.v_cache.copy()
    for i in range(cfg.steps):
        expect_k[:, cfg.T0 + i] = inp.k_new[i]
        expect_v[:, cfg.T0 + i] = inp.v_new[i]
    np.testing.assert_array_equal(bits(kc), expect_k)
    np.testing.assert_array_equal(bits(vc), expect_v)
    assert cl.cpu().numpy().tolist() == [cfg.T0 + cfg.steps] * cfg.B
    for i in sorted(check):
        # oracle step i from the cache state it saw: initial rows + the i rows appended before it
        k_i, v_i = inp.k_cache.copy(), inp.v_cache.copy()
        k_i[:, cfg.T0:cfg.T0 + i] = inp.k_new[:i].transpose(1, 0, 2, 3)
        v_i[:, cfg.T0:cfg.T0 + i] = inp.v_new[:i].transpose(1, 0, 2, 3)
        cl_i = np.full((cfg.B,), cfg.T0 + i, np.int32)
        ro, roc = oracle.decode_step(inp.q_new[i], inp.qc_new[i], inp.k_new[i], inp.v_new[i], k_i, v_i, cl_i,
                                     inp.alpha, inp.beta, inp.alpha_c, inp.beta_c, cfg.window, cfg.scale)
        assert_parity(outs[i][0], ro, f"decode step {i} base")
        assert_parity(outs[i][1], roc, f"decode step {i} copy")
