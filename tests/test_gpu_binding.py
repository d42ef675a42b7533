"""The binding refuses a host tensor among device ones (positions, log-sum-exp, error word)
before anything is launched: a host pointer must never reach a kernel."""
import pytest
import torch

import long_context_attention_orthros_gb300 as orth
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def test_host_positions_lse_and_error_word_are_refused():
    B, T, T_out, Hq, Hkv, d = 1, 64, 2, 4, 2, 64
    bf = dict(dtype=torch.bfloat16, device=dev())
    qc = torch.zeros((B, T_out, Hq, d), **bf)
    k = torch.zeros((B, T, Hkv, d), **bf)
    a = torch.ones((Hq, d), dtype=torch.float32, device=dev())
    pos_host = torch.zeros((B, T_out), dtype=torch.int32)
    with pytest.raises(orth.OrthrosError):
        orth.xattn_fwd(qc, pos_host, k, k, a, a)
    pos = pos_host.to(dev())
    with pytest.raises(orth.OrthrosError):
        orth.xattn_fwd(qc, pos, k, k, a, a, lse=torch.zeros((B, T_out, Hq)))
    with pytest.raises(orth.OrthrosError):
        orth.xattn_fwd(qc, pos, k, k, a, a, dev_err=torch.zeros(1, dtype=torch.int32))
    out = orth.xattn_fwd(qc, pos, k, k, a, a)  # all on the device: accepted
    torch.cuda.synchronize()
    assert out.shape == qc.shape
