"""GPU parity of the fused decode step (append + base SWA + full-cache copy query)
against the fp64 oracle; the KV cache and cache_len must match bit for bit."""
import math

import numpy as np
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
import oracle
from synthetic import CONFIGS, DecodeConfig, bf16_bits, make_decode, reduced
from tests.gpu_util import assert_parity, bf, bits, dev, f32, i32, val

pytestmark = pytest.mark.gpu


class GpuDecode:
    def __init__(self, inp):
        c = inp.cfg
        self.inp = inp
        self.kc, self.vc = bf(inp.k_cache), bf(inp.v_cache)
        self.cl = i32(inp.cache_len)
        self.a, self.b, self.ac, self.bc = (f32(x) for x in (inp.alpha, inp.beta, inp.alpha_c, inp.beta_c))
        self.ws = orth._binding.decode_workspace(c.B, c.L_max, c.Hq, c.Hkv, c.d, dev())
        self.err = torch.zeros(1, dtype=torch.int32, device=dev())

    def step(self, i, qc_override=None):
        inp, c = self.inp, self.inp.cfg
        qc = inp.qc_new[i] if qc_override is None else qc_override
        return orth.decode_step(bf(inp.q_new[i]), bf(qc), bf(inp.k_new[i]), bf(inp.v_new[i]),
                                self.kc, self.vc, self.cl, self.a, self.b, self.ac, self.bc,
                                window=c.window, scale=c.scale, workspace=self.ws, dev_err=self.err)


def _oracle_steps(inp, steps):
    c = inp.cfg
    kc, vc, cl = inp.k_cache.copy(), inp.v_cache.copy(), inp.cache_len.copy()
    outs = []
    for i in steps:
        o, oc = oracle.decode_step(inp.q_new[i], inp.qc_new[i], inp.k_new[i], inp.v_new[i], kc, vc,
                                   cl, inp.alpha, inp.beta, inp.alpha_c, inp.beta_c, c.window, c.scale)
        outs.append((o, oc))
    return outs, kc, vc, cl


@pytest.mark.parametrize("B,T0,steps,Hq,Hkv,d,w", [
    (2, 1000, 6, 32, 8, 128, 128),   # 8B-class heads; crosses a 64-key block boundary
    (1, 63, 3, 8, 2, 128, 128),      # cache shorter than one block
    (2, 130, 4, 4, 4, 64, 128),      # G=1, d=64
    (1, 2000, 3, 16, 1, 128, 7),     # G=16, narrow window
    (1, 1, 2, 8, 2, 128, 128),       # almost empty cache
    (1, 0, 2, 8, 2, 128, 128),       # empty cache: the first token attends to itself only
])
def test_decode_steps_match_oracle(B, T0, steps, Hq, Hkv, d, w):
    cfg = DecodeConfig("case", B=B, T0=T0, steps=steps, Hq=Hq, Hkv=Hkv, d=d, window=w)
    inp = make_decode(cfg, 300 + T0)
    g = GpuDecode(inp)
    ref, kc, vc, cl = _oracle_steps(inp, range(steps))
    for i in range(steps):
        o, oc = g.step(i)
        assert_parity(val(o), ref[i][0], f"step {i} base")
        assert_parity(val(oc), ref[i][1], f"step {i} copy")
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    np.testing.assert_array_equal(bits(g.kc), kc)
    np.testing.assert_array_equal(bits(g.vc), vc)
    np.testing.assert_array_equal(g.cl.cpu().numpy(), cl)


def test_decode_copy_is_isolated_from_cache_and_base():
    """Changing the copy's query changes only oc: o, the cache and cache_len are
    bit-identical (copies never write K/V)."""
    cfg = DecodeConfig("iso", B=2, T0=700, steps=1, Hq=32, Hkv=8, d=128)
    inp = make_decode(cfg, 11)
    res = []
    for qc in (inp.qc_new[0], inp.qc_new[0] ^ np.uint16(0x0001)):
        g = GpuDecode(inp)
        o, oc = g.step(0, qc_override=qc)
        res.append((bits(o), bits(oc), bits(g.kc), bits(g.vc), g.cl.cpu().numpy()))
    for i in (0, 2, 3, 4):
        np.testing.assert_array_equal(res[0][i], res[1][i])


@pytest.mark.parametrize("lens,Hq,Hkv,d,w,steps", [
    ((0, 1, 63, 127, 128, 1000, 4097, 9000), 32, 8, 128, 128, 3),  # B=8, 8B-class heads, ragged
    ((5000, 64, 130, 2), 8, 2, 64, 100, 2),                          # d=64, one sequence far longer
])
def test_decode_ragged_batch_matches_oracle(lens, Hq, Hkv, d, w, steps):
    """Sequences of different cache lengths in one launch: each reads its own cache_len[b]; rows at
    or beyond it hold bf16 NaN, so a read past a sequence's end shows as a non-finite output."""
    B = len(lens)
    cfg = DecodeConfig("ragged", B=B, T0=max(lens), steps=steps, Hq=Hq, Hkv=Hkv, d=d, window=w)
    inp = make_decode(cfg, 4242 + B)
    for b, n in enumerate(lens):
        inp.k_cache[b, n:] = cfg.fill_unused
        inp.v_cache[b, n:] = cfg.fill_unused
    inp.cache_len[:] = np.asarray(lens, np.int32)
    g = GpuDecode(inp)
    ref, kc, vc, cl = _oracle_steps(inp, range(steps))
    for i in range(steps):
        o, oc = g.step(i)
        assert_parity(val(o), ref[i][0], f"ragged step {i} base")
        assert_parity(val(oc), ref[i][1], f"ragged step {i} copy")
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    np.testing.assert_array_equal(bits(g.kc), kc)
    np.testing.assert_array_equal(bits(g.vc), vc)
    np.testing.assert_array_equal(g.cl.cpu().numpy(), np.asarray(lens, np.int32) + steps)


def test_decode_equals_prefill_exactly_on_one_hot_values():
    """With K = 0 every logit is 0, so each softmax weight is exactly 1 and o = (sum of the attended
    V rows) / (their count).  With V row j = e_(j mod d) the output is count_c / n per column, a
    value each kernel reaches exactly up to its final bf16 rounding, and one key row too many or
    too few moves a column by 1/n, far beyond that rounding.  Decode at position p and the
    prefill kernels at p must both give the closed form: the decode-equals-prefill invariant
    with the mask checked row for row."""
    B, Hq, Hkv, d, w = 2, 8, 2, 128, 128
    for p in (0, 5, 127, 128, 129, 1000, 4000):
        T = p + 1
        cfg = DecodeConfig("onehot", B=B, T0=p, steps=1, Hq=Hq, Hkv=Hkv, d=d, window=w)
        inp = make_decode(cfg, 77)
        onehot = np.zeros((T, d), np.float32)
        onehot[np.arange(T), np.arange(T) % d] = 1.0
        vrows = np.broadcast_to(bf16_bits(onehot)[None, :, None, :], (B, T, Hkv, d))
        inp.k_cache[:, :p] = 0
        inp.v_cache[:, :p] = vrows[:, :p]
        inp.k_new[0] = 0
        inp.v_new[0] = vrows[:, p]
        g = GpuDecode(inp)
        o, oc = g.step(0)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0

        def closed_form(lo):
            cnt = np.zeros(d)
            np.add.at(cnt, np.arange(lo, T) % d, 1.0)
            return np.broadcast_to(cnt / (T - lo), (B, Hq, d))
        want_o, want_oc = closed_form(max(0, p - w + 1)), closed_form(0)
        k_full = bits(g.kc)[:, :T]
        v_full = bits(g.vc)[:, :T]
        q = np.zeros((B, T, Hq, d), np.uint16)
        q[:, p] = inp.q_new[0]
        o_pre = val(orth.swa_fwd(bf(q), bf(k_full), bf(v_full), g.a, g.b, window=w))[:, p]
        oc_pre = val(orth.xattn_fwd(bf(inp.qc_new[0][:, None]), i32(np.full((B, 1), p, np.int32)),
                                    bf(k_full), bf(v_full), g.ac, g.bc))[:, 0]
        for got, want, what in ((val(o), want_o, "decode base"), (o_pre, want_o, "prefill base"),
                                (val(oc), want_oc, "decode copy"), (oc_pre, want_oc, "prefill copy")):
            assert np.abs(got - want).max() <= 2.0 ** -8 * np.abs(want).max() + 1e-7, (p, what)


def test_decode_equals_prefill_at_appended_position():
    """Decode of token p after a prefix equals the prefill kernels' result at p."""
    B, T, Hq, Hkv, d, w = 1, 800, 8, 2, 128, 128
    cfg = DecodeConfig("dp", B=B, T0=T - 1, steps=1, Hq=Hq, Hkv=Hkv, d=d, window=w)
    inp = make_decode(cfg, 12)
    g = GpuDecode(inp)
    o, oc = g.step(0)
    k_full = bits(g.kc)[:, :T]
    v_full = bits(g.vc)[:, :T]
    q = np.zeros((B, T, Hq, d), np.uint16)
    q[:, T - 1] = inp.q_new[0]
    o_pre = orth.swa_fwd(bf(q), bf(k_full), bf(v_full), g.a, g.b, window=w)
    oc_pre = orth.xattn_fwd(bf(inp.qc_new[0][:, None]), i32(np.full((B, 1), T - 1, np.int32)),
                            bf(k_full), bf(v_full), g.ac, g.bc)
    assert np.abs(val(o) - val(o_pre)[:, T - 1]).max() <= 1e-2
    assert np.abs(val(oc) - val(oc_pre)[:, 0]).max() <= 1e-2


def test_decode_full_cache_sets_error_and_leaves_cache():
    cfg = DecodeConfig("fullc", B=2, T0=10, steps=1, Hq=8, Hkv=2, d=128)
    inp = make_decode(cfg, 13)
    inp.cache_len[1] = cfg.L_max  # sequence 1 is full
    g = GpuDecode(inp)
    before = bits(g.kc).copy()
    o, oc = g.step(0)
    torch.cuda.synchronize()
    assert int(g.err.item()) & orth.DEVERR_CACHE_FULL
    assert (val(o)[1] == 0).all() and (val(oc)[1] == 0).all()
    after = bits(g.kc)
    np.testing.assert_array_equal(after[1], before[1])
    assert g.cl.cpu().numpy().tolist() == [11, cfg.L_max]


def test_decode_steps_replay_as_one_cuda_graph():
    """Multi-step decode captured once as a CUDA graph: the step allocates nothing, never
    waits on the host and keeps cache_len on the device, so replaying the captured steps
    gives the eager steps' outputs and cache bit for bit (and meets the oracle)."""
    cfg = DecodeConfig("graph", B=2, T0=700, steps=8, Hq=32, Hkv=8, d=128)
    inp = make_decode(cfg, 911)
    qn, qcn, kn, vn = bf(inp.q_new), bf(inp.qc_new), bf(inp.k_new), bf(inp.v_new)

    def run(graph):
        g = GpuDecode(inp)
        o = torch.empty((cfg.B, cfg.Hq, cfg.d), dtype=torch.bfloat16, device=dev())
        oc = torch.empty_like(o)
        outs = [torch.empty_like(o) for _ in range(cfg.steps)], [torch.empty_like(o) for _ in range(cfg.steps)]

        def steps():
            for i in range(cfg.steps):
                orth.decode_step(qn[i], qcn[i], kn[i], vn[i], g.kc, g.vc, g.cl, g.a, g.b, g.ac, g.bc,
                                 window=cfg.window, scale=cfg.scale, o=o, oc=oc, workspace=g.ws, dev_err=g.err)
                outs[0][i].copy_(o)
                outs[1][i].copy_(oc)
        if graph:
            cl0 = g.cl.clone()
            kc0, vc0 = g.kc.clone(), g.vc.clone()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                steps()  # warm-up on a side stream (sets kernel attributes)
            torch.cuda.current_stream().wait_stream(s)
            g.cl.copy_(cl0)
            g.kc.copy_(kc0)
            g.vc.copy_(vc0)
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg):
                steps()
            g.cl.copy_(cl0)  # capture does not run the steps; start from the initial state
            g.kc.copy_(kc0)
            g.vc.copy_(vc0)
            cg.replay()
        else:
            steps()
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        return g, outs

    ge, oe = run(False)
    gg, og = run(True)
    assert torch.equal(ge.cl, gg.cl)
    assert torch.equal(ge.kc.view(torch.int16), gg.kc.view(torch.int16))
    assert torch.equal(ge.vc.view(torch.int16), gg.vc.view(torch.int16))
    for i in range(cfg.steps):
        assert torch.equal(oe[0][i].view(torch.int16), og[0][i].view(torch.int16))
        assert torch.equal(oe[1][i].view(torch.int16), og[1][i].view(torch.int16))
    ref, _kc, _vc, _cl = _oracle_steps(inp, range(cfg.steps))
    for i in (0, cfg.steps - 1):
        assert_parity(val(og[0][i]), ref[i][0], f"graph step {i} base")
        assert_parity(val(og[1][i]), ref[i][1], f"graph step {i} copy")
