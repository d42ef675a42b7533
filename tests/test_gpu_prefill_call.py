"""GPU parity of the one-call prefill layer (orthros_prefill_fwd) against the fp64
oracle: the base stream (Eq. 4) and the output copies (Eq. 5) of one call.  Both
outputs must also equal separate orthros_swa_fwd / orthros_xattn_fwd calls bit for bit
(for few copies the call runs the copies' pass on a second stream beside the SWA
kernel, which holds fewer SMs; neither changes any result)."""
import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import PrefillConfig, make_prefill
from tests.gpu_util import assert_parity, bf, dev, f32, i32, val

pytestmark = pytest.mark.gpu


def _run(inp, window=None):
    cfg = inp.cfg
    w = cfg.window if window is None else window
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q_all = bf(inp.q_raw)
    k, v = bf(inp.k), bf(inp.v)
    qc = q_all[:, cfg.T:] if cfg.appended else bf(inp.qc_raw)
    o, oc = orth.prefill_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), qc, i32(inp.pos), f32(inp.alpha_c),
                             f32(inp.beta_c), window=w, scale=cfg.scale, dev_err=err)
    o_swa = orth.swa_fwd(q_all, k, v, f32(inp.alpha), f32(inp.beta), window=w, scale=cfg.scale, dev_err=err)
    oc_x = orth.xattn_fwd(qc, i32(inp.pos), k, v, f32(inp.alpha_c), f32(inp.beta_c), scale=cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert torch.equal(oc.view(torch.int16), oc_x.view(torch.int16)), "copy output differs from xattn_fwd"
    return o, oc, o_swa, int(err.item())


def _check(inp, window=None):
    cfg = inp.cfg
    w = cfg.window if window is None else window
    o, oc, o_swa, err = _run(inp, window)
    assert err == 0
    assert torch.equal(o.view(torch.int16), o_swa.view(torch.int16)), "base output differs from swa_fwd"
    ref_o = oracle.swa(np.ascontiguousarray(inp.q_base), inp.k, inp.v, inp.alpha, inp.beta, w, cfg.scale)
    ref_oc = oracle.xattn(np.ascontiguousarray(inp.qc_raw), inp.pos, inp.k, inp.v, inp.alpha_c, inp.beta_c,
                          cfg.scale)
    assert_parity(val(o), ref_o, "base O")
    assert_parity(val(oc), ref_oc, "copy O'")


def _positions(cfg, seed):
    """Seeded original positions: block edges, the ends, duplicates and random rows."""
    g = np.random.default_rng(seed)
    edges = np.array([0, 31, 32, 63, 64, cfg.T - 1, cfg.T - 1, cfg.T // 2], np.int64)
    pos = np.empty((cfg.B, cfg.T_out), np.int32)
    for b in range(cfg.B):
        cand = np.concatenate([edges[edges < cfg.T], g.integers(0, cfg.T, size=cfg.T_out)])
        pos[b] = g.permutation(cand)[:cfg.T_out]
    return pos


@pytest.mark.parametrize("B,T,Hq,Hkv,d,T_out", [
    (2, 1000, 32, 8, 128, 1),   # 8B-class heads, one copy (the prefill workload's shape)
    (1, 20000, 32, 8, 128, 1),  # one sequence (the 1M workload's layout), copies beside SWA
    (2, 1000, 32, 8, 128, 4),   # 16 copy rows per KV head
    (1, 777, 8, 4, 64, 3),      # G=2, d=64
    (1, 257, 16, 2, 128, 2),    # G=8
    (1, 200, 16, 1, 64, 1),     # G=16
    (3, 5000, 8, 2, 128, 2),    # each stream spread over many CTAs
    (1, 5, 4, 1, 128, 2),       # fewer tiles than SMs
    (2, 1000, 32, 8, 128, 8),   # 32 copy rows per KV head
    (1, 3000, 16, 2, 128, 1),   # G=8, one copy
    (2, 4097, 8, 4, 128, 4),    # G=2, 8 copy rows, T off the tile grid
    (1, 300, 16, 2, 64, 1),     # d=64, G=8
    (4, 9000, 32, 8, 128, 2),   # 8 copy rows of 8B-class heads, streams over many CTAs
    (2, 3000, 8, 8, 128, 3),    # G=1: the copies' pass beside SWA on more SMs (its share of bytes is larger)
    (1, 6000, 8, 4, 64, 4),     # G=2, d=64, 8 copy rows
])
def test_prefill_call_parity(B, T, Hq, Hkv, d, T_out):
    cfg = PrefillConfig("call", B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, T_out=T_out)
    inp = make_prefill(cfg, 2000 + T + T_out)
    inp.pos[:] = _positions(cfg, T + 7 * T_out)
    _check(inp)


def test_prefill_call_last_position_appended():
    """Algorithm 2's layout: the copy of the last position stored after the base tokens."""
    cfg = PrefillConfig("call_app", B=2, T=2048, Hq=32, Hkv=8, d=128, T_out=1, appended=True)
    _check(make_prefill(cfg, 31))


def test_prefill_call_wide_window():
    """A band wider than tensor memory holds (the streaming SWA kernel)."""
    cfg = PrefillConfig("call_wide", B=1, T=700, Hq=8, Hkv=2, d=128, window=600, T_out=2)
    inp = make_prefill(cfg, 44)
    _check(inp, window=600)


def test_prefill_call_bad_position():
    cfg = PrefillConfig("call_bad", B=1, T=600, Hq=8, Hkv=2, d=128, T_out=3)
    inp = make_prefill(cfg, 45)
    inp.pos[0] = [100, 600, -1]
    o, oc, o_swa, err = _run(inp)
    assert err & orth.DEVERR_POSITION
    got = val(oc)
    assert (got[0, 1] == 0).all() and (got[0, 2] == 0).all()
    ref = oracle.xattn(np.ascontiguousarray(inp.qc_raw[:, :1]), inp.pos[:, :1], inp.k, inp.v, inp.alpha_c,
                       inp.beta_c, cfg.scale)
    assert_parity(got[:, :1], ref, "valid copy next to bad ones")
    assert torch.equal(o.view(torch.int16), o_swa.view(torch.int16))


@pytest.mark.parametrize("T,Hq,Hkv", [(600, 8, 2), (5000, 16, 2)])
def test_prefill_call_bad_and_early_positions(T, Hq, Hkv):
    """An out-of-range position gets zeros and the position flag; copies at position 0 and in
    the first window meet the oracle."""
    cfg = PrefillConfig("call_bad1", B=2, T=T, Hq=Hq, Hkv=Hkv, d=128, T_out=8 // (Hq // Hkv))
    inp = make_prefill(cfg, 46 + T)
    inp.pos[:] = np.array([[0, -1], [T, 37]] if cfg.T_out == 2 else [[-5], [T - 1]], np.int32)
    o, oc, o_swa, err = _run(inp)
    assert err & orth.DEVERR_POSITION
    assert torch.equal(o.view(torch.int16), o_swa.view(torch.int16))
    got = val(oc)
    valid = (inp.pos >= 0) & (inp.pos < T)
    assert (got[~valid] == 0).all()
    for b in range(cfg.B):
        for i in range(cfg.T_out):
            if valid[b, i]:
                ref = oracle.xattn(np.ascontiguousarray(inp.qc_raw[b:b + 1, i:i + 1]),
                                   np.ascontiguousarray(inp.pos[b:b + 1, i:i + 1]), inp.k[b:b + 1], inp.v[b:b + 1],
                                   inp.alpha_c, inp.beta_c, cfg.scale)
                assert_parity(got[b:b + 1, i:i + 1], ref, f"copy ({b}, {i})")


def test_prefill_call_stream_order():
    """Back-to-back calls with K rewritten on the caller's stream between them: the copies'
    pass (on the second stream) of each call sees the K of its own call."""
    cfg = PrefillConfig("call_order", B=2, T=4096, Hq=32, Hkv=8, d=128, T_out=1)
    inp = make_prefill(cfg, 47)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q, k, v = bf(inp.q_raw), bf(inp.k), bf(inp.v)
    qc, pos = bf(inp.qc_raw), i32(inp.pos)
    a, b, ac, bc = f32(inp.alpha), f32(inp.beta), f32(inp.alpha_c), f32(inp.beta_c)
    outs = []
    for it in range(3):
        o, oc = orth.prefill_fwd(q, k, v, a, b, qc, pos, ac, bc, window=cfg.window, scale=cfg.scale, dev_err=err)
        outs.append((o, oc, k.clone()))
        k.mul_(-1.0)  # on the caller's stream, right behind the call
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for o, oc, kk in outs:
        o_ref = orth.swa_fwd(q, kk, v, a, b, window=cfg.window, scale=cfg.scale)
        oc_ref = orth.xattn_fwd(qc, pos, kk, v, ac, bc, scale=cfg.scale)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(oc.view(torch.int16), oc_ref.view(torch.int16))


def test_prefill_call_cuda_graph():
    """The call captured in a CUDA graph (its second stream joins the capture) and replayed
    gives the eager call's bits."""
    cfg = PrefillConfig("call_graph", B=2, T=4096, Hq=32, Hkv=8, d=128, T_out=1)
    inp = make_prefill(cfg, 48)
    q, k, v = bf(inp.q_raw), bf(inp.k), bf(inp.v)
    qc, pos = bf(inp.qc_raw), i32(inp.pos)
    a, b, ac, bc = f32(inp.alpha), f32(inp.beta), f32(inp.alpha_c), f32(inp.beta_c)
    ws = torch.empty(max(orth.prefill_workspace_size(cfg.B, cfg.T, cfg.T_out, cfg.Hq, cfg.Hkv, cfg.d), 256),
                     dtype=torch.uint8, device=dev())
    o = torch.empty((cfg.B, cfg.T, cfg.Hq, cfg.d), dtype=torch.bfloat16, device=dev())
    oc = torch.empty((cfg.B, cfg.T_out, cfg.Hq, cfg.d), dtype=torch.bfloat16, device=dev())
    o_e, oc_e = orth.prefill_fwd(q, k, v, a, b, qc, pos, ac, bc, window=cfg.window, scale=cfg.scale)
    s = torch.cuda.Stream(dev())
    s.wait_stream(torch.cuda.current_stream(dev()))
    with torch.cuda.stream(s):  # warm the call on the capture stream
        orth.prefill_fwd(q, k, v, a, b, qc, pos, ac, bc, window=cfg.window, scale=cfg.scale, out=o, out_c=oc,
                         workspace=ws)
    torch.cuda.current_stream(dev()).wait_stream(s)
    torch.cuda.synchronize()
    o.zero_()
    oc.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        orth.prefill_fwd(q, k, v, a, b, qc, pos, ac, bc, window=cfg.window, scale=cfg.scale, out=o, out_c=oc,
                         workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_e.view(torch.int16))
    assert torch.equal(oc.view(torch.int16), oc_e.view(torch.int16))
