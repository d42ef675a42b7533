"""C ABI checks that need no GPU: the library builds, loads, exports every
function include/orthros.h declares, and its host-side argument checks and
workspace-size queries behave as documented (none of these calls touches a GPU).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "orthros.h")


@pytest.fixture(scope="module")
def L():
    from long_context_attention_orthros_gb300 import build
    build.build()
    import long_context_attention_orthros_gb300 as orth
    return orth.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(orthros_\w+)\s*\(", text)))


def test_header_declares_the_operator_entry_points():
    names = _declared()
    for n in ("orthros_swa_fwd", "orthros_xattn_fwd", "orthros_decode_step",
              "orthros_xattn_workspace_size", "orthros_decode_workspace_size",
              "orthros_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_status_strings(L):
    assert L.orthros_status_string(0) == b"ok"
    assert L.orthros_status_string(3).startswith(b"workspace")
    assert L.orthros_status_string(99) == b"unknown status"
    assert L.orthros_version() >= 100


def _aligned_dummy():
    # an aligned host address that is never dereferenced: every call below fails a
    # host-side check before any pointer is used or any CUDA call is made
    buf = (ctypes.c_uint8 * 64)()
    return ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15), buf


def test_swa_rejects_bad_arguments_on_the_host(L):
    p, _keep = _aligned_dummy()
    args = dict(B=1, T=16, Hq=4, Hkv=2, d=128, w=8)

    def call(**kw):
        a = {**args, **kw}
        return L.orthros_swa_fwd(kw.get("q", p), p, p, p, p, p, a["B"], a["T"], a["Hq"], a["Hkv"],
                                 a["d"], a["w"], ctypes.c_float(0.1), 0, 0, 0, None, None)
    assert call(q=None) == 1
    assert call(q=ctypes.c_void_p(p.value + 2)) == 1  # misaligned
    assert call(B=0) == 1
    assert call(T=0) == 1
    assert call(w=0) == 1
    assert call(d=96) == 2
    assert call(Hq=6, Hkv=4) == 2
    assert call(Hq=96, Hkv=3) == 2  # 32 heads per KV head: unsupported grouping
    assert L.orthros_swa_fwd(p, p, p, p, p, p, 1, 16, 4, 2, 128, 8, ctypes.c_float(0.1), 3, 0, 0,
                             None, None) == 1  # batch stride below dense
    assert L.orthros_swa_fwd(p, p, p, p, p, p, 1, 16, 4, 2, 128, 8, ctypes.c_float(float("nan")), 0,
                             0, 0, None, None) == 1


def test_xattn_workspace_size_and_checks(L):
    p, _keep = _aligned_dummy()
    assert L.orthros_xattn_workspace_size(1, 1, 0, 4, 2, 128) == 0
    assert L.orthros_xattn_workspace_size(1, 1, 100, 4, 2, 100) == 0
    small = L.orthros_xattn_workspace_size(2, 1, 131072, 32, 8, 128)
    assert small > 0
    # more copies need more partial-result space
    assert L.orthros_xattn_workspace_size(4, 2048, 16384, 32, 8, 128) > 0
    # T_out == 0 is a no-op that never touches memory
    assert L.orthros_xattn_fwd(None, None, None, None, None, None, None, 1, 0, 10, 4, 2, 128,
                               ctypes.c_float(0.1), 0, 0, 0, None, 0, None, None) == 0
    # workspace too small
    assert L.orthros_xattn_fwd(p, p, p, p, p, p, p, 2, 1, 131072, 32, 8, 128, ctypes.c_float(0.1),
                               0, 0, 0, p, 16, None, None) == 3
    assert L.orthros_xattn_fwd(p, p, p, p, p, p, p, 2, 1, 131072, 32, 8, 128, ctypes.c_float(0.1),
                               0, 0, 0, None, small, None, None) == 3
    # the log-sum-exp variant: a misaligned lse is rejected before anything runs
    assert L.orthros_xattn_fwd_lse(p, p, p, p, p, p, p, ctypes.c_void_p(p.value + 4), 2, 1, 131072, 32, 8, 128,
                                   ctypes.c_float(0.1), 0, 0, 0, p, small, None, None) == 1
    assert L.orthros_xattn_fwd_lse(p, p, p, p, p, p, p, p, 2, 1, 131072, 32, 8, 128, ctypes.c_float(0.1),
                                   0, 0, 0, p, 16, None, None) == 3


def test_decode_workspace_size_and_checks(L):
    p, _keep = _aligned_dummy()
    n = L.orthros_decode_workspace_size(2, 131200, 32, 8, 128)
    assert n > 0
    assert L.orthros_decode_workspace_size(2, 0, 32, 8, 128) == 0
    assert L.orthros_decode_step(p, p, p, p, p, p, p, 131200, p, p, p, p, p, p, 2, 32, 8, 128, 128,
                                 ctypes.c_float(0.1), p, 8, None, None) == 3
    assert L.orthros_decode_step(p, p, p, p, p, p, None, 131200, p, p, p, p, p, p, 2, 32, 8, 128,
                                 128, ctypes.c_float(0.1), p, n, None, None) == 1


def test_swa_bwd_workspace_size_and_checks(L):
    p, _keep = _aligned_dummy()
    n = L.orthros_swa_bwd_workspace_size(2, 1000, 32, 8, 128)
    nkb = (1000 + 63) // 64  # 64-key blocks
    # lse, D; fp16 K; each key row's shift (int8, whole blocks); each block's flag; fp16 q
    # (every part here is already a multiple of 256 bytes)
    assert n == (2 * 4 * 2 * 1000 * 32 + 2 * 2 * 1000 * 8 * 128 + 2 * 8 * nkb * 64 + 256 +
                 2 * 2 * 1000 * 32 * 128)
    assert L.orthros_swa_bwd_workspace_size(2, 1000, 32, 8, 96) == 0
    assert L.orthros_swa_bwd_workspace_size(0, 1000, 32, 8, 128) == 0

    def call(w=128, ws=p, nbytes=n, q=p, d=128):
        return L.orthros_swa_bwd(q, p, p, p, p, p, p, None, p, p, p, p, p, 2, 1000, 32, 8, d, w,
                                 ctypes.c_float(0.1), ws, nbytes, None, None)
    assert call(q=None) == 1
    assert call(w=0) == 1
    assert call(d=96) == 2
    assert call(q=ctypes.c_void_p(p.value + 4)) == 1  # misaligned


def test_xattn_bwd_workspace_size_and_checks(L):
    p, _keep = _aligned_dummy()
    n = L.orthros_xattn_bwd_workspace_size(4, 2048, 16384, 32, 8, 128)
    # row lse and D, fp16 K, key-row shifts and block flags (16384 keys: 256 blocks), split
    # partials, the copies' fp16 q
    assert n == (2 * 4 * 4 * 2048 * 32 + 2 * 4 * 16384 * 8 * 128 + 4 * 8 * 16384 + 4 * 8 * 256 +
                 4 * 8 * 64 * 128 * 8 + 2 * 4 * 2048 * 32 * 128)
    assert L.orthros_xattn_bwd_workspace_size(4, 2048, 0, 32, 8, 128) == 0
    assert L.orthros_xattn_bwd_workspace_size(4, 2048, 16384, 32, 8, 96) == 0

    def call(ws=p, nbytes=n, pos=p, T_out=2048, Hkv=8, lse=None):
        return L.orthros_xattn_bwd(p, pos, p, p, p, p, p, p, lse, p, p, p, p, p, 4, T_out, 16384, 32, Hkv, 128,
                                   ctypes.c_float(0.1), 1, ws, nbytes, None, None)
    assert call(pos=None) == 1
    assert call(lse=ctypes.c_void_p(p.value + 4)) == 1  # misaligned log-sum-exp
    assert call(T_out=-1) == 1
    assert call(Hkv=5) == 2
    assert call(ws=None) == 3
    assert call(nbytes=n - 4) == 3
    assert call(ws=None) == 3
    assert call(nbytes=n - 4) == 3


def test_attn_bwd_workspace_size_and_checks(L):
    p, _keep = _aligned_dummy()
    n = L.orthros_attn_bwd_workspace_size(2, 1000, 64, 32, 8, 128)
    base = L.orthros_swa_bwd_workspace_size(2, 1000, 32, 8, 128)
    # the base stream's region (256-aligned), then the copies' rows, split partials and fp16 q
    copies = ((8 * 2 * 64 * 32 + 255) // 256 * 256) + 2 * 8 * 64 * 128 * 8 + 2 * 2 * 64 * 32 * 128
    assert n == (base + 255) // 256 * 256 + copies
    assert L.orthros_attn_bwd_workspace_size(2, 1000, 0, 32, 8, 128) > base
    assert L.orthros_attn_bwd_workspace_size(2, 0, 64, 32, 8, 128) == 0
    assert L.orthros_attn_bwd_workspace_size(2, 1000, -1, 32, 8, 128) == 0
    assert L.orthros_attn_bwd_workspace_size(2, 1000, 64, 32, 5, 128) == 0

    def call(ws=p, nbytes=n, pos=p, T_out=64, Hkv=8, window=128, lsec=None):
        args = [p] * 9 + [pos] + [p] * 4 + [lsec] + [p] * 8
        return L.orthros_attn_bwd(*args, 2, 1000, T_out, 32, Hkv, 128, window, ctypes.c_float(0.1), ws, nbytes,
                                  None, None)
    assert call(pos=None) == 1
    assert call(window=0) == 1
    assert call(T_out=-1) == 1
    assert call(lsec=ctypes.c_void_p(p.value + 4)) == 1
    assert call(Hkv=5) == 2
    assert call(ws=None) == 3
    assert call(nbytes=n - 4) == 3


def test_a_c99_program_links_and_calls_the_library(tmp_path):
    """The boundary as a C caller sees it: the header compiles as strict C99, a program links
    against the shared library and calls its host-only entry points (version, status strings,
    workspace sizes), whose values agree with those seen through the binding."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    import long_context_attention_orthros_gb300 as orth
    libpath = orth.library_path
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include "orthros.h"
int main(void)
{
    printf("%d\n", orthros_version());
    printf("%s\n", orthros_status_string(ORTHROS_ERR_WORKSPACE));
    printf("%zu\n", orthros_attn_bwd_workspace_size(2, 1000, 64, 32, 8, 128));
    printf("%zu\n", orthros_xattn_workspace_size(2, 1, 131072, 32, 8, 128));
    printf("%zu\n", orthros_decode_workspace_size(2, 131200, 32, 8, 128));
    return orthros_swa_bwd_workspace_size(0, 1, 1, 1, 64) == 0 ? 0 : 1;
}
""")
    exe = tmp_path / "caller"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    libdir = os.path.dirname(libpath)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", f"-I{inc}", str(src), "-o", str(exe),
                    f"-L{libdir}", "-l:" + os.path.basename(libpath), f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert int(out[0]) > 0
    assert out[1] == "workspace missing or too small"
    assert int(out[2]) == orth.attn_bwd_workspace_size(2, 1000, 64, 32, 8, 128)
    assert int(out[3]) == orth.xattn_workspace_size(2, 1, 131072, 32, 8, 128)
    assert int(out[4]) == orth.decode_workspace_size(2, 131200, 32, 8, 128)
