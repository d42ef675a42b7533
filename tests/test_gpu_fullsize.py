"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times, against the fp64 oracle on sampled outputs the oracle computes one by one:
the 8B-class 128K prefill (B=2), the 1M-token prefill with scaled key rows, the
SFT layer with 2048 appended shuffled copies per sequence, and 128 decode steps
after a 131072-token cache."""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import CONFIGS, SEEDS, make_decode, make_prefill
from tests.gpu_util import assert_parity, bf, bits, dev, f32, i32, val

pytestmark = pytest.mark.gpu


def _sample_rows(cfg, n, seed):
    """Seeded (b, t) rows: the first window, the tail, and random rows in between."""
    g = np.random.default_rng(seed)
    t = np.concatenate([np.arange(0, 160, 7), np.arange(cfg.T - 40, cfg.T),
                        g.integers(0, cfg.T, size=n)])
    b = g.integers(0, cfg.B, size=t.size)
    return b.astype(np.int32), t.astype(np.int32)


def _prefill_full(name, n_rows, copies=None):
    cfg = CONFIGS[name]
    inp = make_prefill(cfg, SEEDS[cfg.name])
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q_all = bf(inp.q_raw)
    k, v = bf(inp.k), bf(inp.v)
    o = orth.swa_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), window=cfg.window, scale=cfg.scale,
                     dev_err=err)
    qc = q_all[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    oc = orth.xattn_fwd(qc, i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale,
                        dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bi, ti = _sample_rows(cfg, n_rows, 7)
    got = val(o[torch.from_numpy(bi).long().to(dev()), torch.from_numpy(ti).long().to(dev())])
    ref = oracle.swa_rows(inp.q_base, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale, bi, ti)
    assert_parity(got, ref, f"{name} base rows")
    sel = np.arange(cfg.T_out) if copies is None else copies
    ref_c = oracle.xattn(np.ascontiguousarray(inp.qc_raw[:, sel]), np.ascontiguousarray(inp.pos[:, sel]),
                         inp.k, inp.v, inp.alpha_c, inp.beta_c, cfg.scale)
    assert_parity(val(oc)[:, sel], ref_c, f"{name} copies")
    return inp, o


def test_prefill_128k_full_size():
    _prefill_full("prefill_128k", 2048)


def test_prefill_1m_needles_full_size():
    inp, o = _prefill_full("prefill_1m", 1024)
    # rows whose window holds a scaled key row
    cfg = inp.cfg
    nd = inp.needles[(inp.needles > 200) & (inp.needles < cfg.T - 200)][:16]
    ti = (nd[:, None] + np.array([0, 5, 63, 127])[None, :]).reshape(-1).astype(np.int32)
    bi = np.zeros_like(ti)
    got = val(o[torch.from_numpy(bi).long().to(dev()), torch.from_numpy(ti).long().to(dev())])
    ref = oracle.swa_rows(inp.q_base, inp.k, inp.v, inp.alpha, inp.beta, cfg.window, cfg.scale, bi, ti)
    assert_parity(got, ref, "1M rows next to scaled keys")


def test_sft_16k_full_size():
    g = np.random.default_rng(11)
    _prefill_full("sft_16k", 1024, copies=np.sort(g.choice(2048, size=24, replace=False)))


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
