"""The Python binding marshals arguments only: every entry point refuses host (CPU) tensors
with OrthrosError instead of computing anything itself, so there is no CPU fallback.  Runs
without a GPU (the checks come before any library call)."""
import pytest
import torch

import long_context_attention_orthros_gb300 as orth

B, T, T_out, Hq, Hkv, d = 1, 8, 2, 4, 2, 64


def _bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def _f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def _args():
    return dict(q=_bf(B, T, Hq, d), k=_bf(B, T, Hkv, d), v=_bf(B, T, Hkv, d), a=_f32(Hq, d), b=_f32(Hq, d),
                o=_bf(B, T, Hq, d), dO=_bf(B, T, Hq, d), qc=_bf(B, T_out, Hq, d),
                pos=torch.zeros((B, T_out), dtype=torch.int32), oc=_bf(B, T_out, Hq, d), dOc=_bf(B, T_out, Hq, d))


CALLS = {
    "swa_fwd": lambda x: orth.swa_fwd(x["q"], x["k"], x["v"], x["a"], x["b"]),
    "swa_fwd_lse": lambda x: orth.swa_fwd_lse(x["q"], x["k"], x["v"], x["a"], x["b"]),
    "swa_fwd_rows": lambda x: orth.swa_fwd_rows(x["q"], x["k"], x["v"], x["a"], x["b"], 0, T),
    "xattn_fwd": lambda x: orth.xattn_fwd(x["qc"], x["pos"], x["k"], x["v"], x["a"], x["b"]),
    "xattn_fwd_lse": lambda x: orth.xattn_fwd(x["qc"], x["pos"], x["k"], x["v"], x["a"], x["b"], lse=True),
    "swa_bwd": lambda x: orth.swa_bwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["o"], x["dO"]),
    "xattn_bwd": lambda x: orth.xattn_bwd(x["qc"], x["pos"], x["k"], x["v"], x["a"], x["b"], x["oc"], x["dOc"]),
    "attn_bwd": lambda x: orth.attn_bwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["o"], x["dO"], x["qc"], x["pos"],
                                        x["a"], x["b"], x["oc"], x["dOc"]),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(orth.OrthrosError):
        CALLS[name](_args())


def test_pointer_marshalling_refuses_host_tensors():
    """Every tensor handed to the library goes through one marshalling helper, which takes
    device tensors of the call's GPU only (a host pointer would reach a kernel otherwise)."""
    from long_context_attention_orthros_gb300._binding import _ptr
    assert _ptr(None) is None
    with pytest.raises(orth.OrthrosError):
        _ptr(torch.zeros(4, dtype=torch.int32))
