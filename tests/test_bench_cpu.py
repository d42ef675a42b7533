"""The benchmark's roofline accounting, on the CPU: the algorithmic byte and pair counts that
roofline.achieved divides by, pinned by brute-force enumeration of what Eqs. (4) and (5) read and
write on small shapes, and the launch counts that gpu_launches claims, against the kernel sequence
the library runs for the benchmark's workloads (the ncu launch list of the bench command)."""
import numpy as np
import pytest

import bench
from synthetic import CONFIGS


@pytest.mark.parametrize("T,w", [(1, 128), (5, 3), (128, 128), (129, 128), (300, 7), (1000, 128)])
def test_swa_pairs_counts_every_row_key_pair_of_the_window(T, w):
    B, Hq = 2, 3
    pairs = sum(1 for t in range(T) for j in range(T) if max(0, t - w + 1) <= j <= t)
    assert bench.swa_pairs(B, T, Hq, w) == B * Hq * pairs


def test_swa_bytes_is_each_input_and_output_once():
    B, T, Hq, Hkv, d = 2, 7, 6, 2, 64
    tensors = {"q": (B, T, Hq, d), "o": (B, T, Hq, d), "k": (B, T, Hkv, d), "v": (B, T, Hkv, d)}
    assert bench.swa_bytes(B, T, Hq, Hkv, d) == sum(2 * int(np.prod(s)) for s in tensors.values())
    # the 8B-class 128K workload: the 5.37 GB one SWA launch is measured against
    assert bench.swa_bytes(2, 131072, 32, 8, 128) == 5368709120


def test_xattn_bytes_reads_keys_up_to_each_sequences_last_copy():
    Hq, Hkv, d, T_kv = 4, 2, 64, 100
    pos = np.array([[3, 17, 5], [99, 0, 42]])
    B, T_out = pos.shape
    key_rows = sum(len(set(j for i in range(T_out) for j in range(pos[b, i] + 1))) for b in range(B))
    expect = key_rows * Hkv * d * 2 * 2 + 2 * B * T_out * Hq * d * 2  # K and V rows; q' and o'
    assert bench.xattn_bytes(pos, Hq, Hkv, d, T_kv) == expect


def test_launch_counts_match_the_kernel_sequence_of_each_workload():
    # prefill at 128K and 1M: the SWA kernel, the copies' pass beside it, the combine of its partials
    assert bench.launches_per_prefill_step(CONFIGS["prefill_128k"]) == 3
    assert bench.launches_per_prefill_step(CONFIGS["prefill_1m"]) == 3
    # SFT layer (2048 copies per sequence): the SWA kernel and the tensor-memory copies kernel
    assert bench.launches_per_prefill_step(CONFIGS["sft_16k"]) == 2
    # layer gradient at the 128K workload (G = 4, w = 128, one copy): fp16 K, the base rows pass,
    # the band dq, the copies' rows pass, the copies' dq, one dK/dV launch
    assert bench.bwd_launches_per_call(1, 4, 128) == 6
