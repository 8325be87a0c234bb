"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host (no GPU needed: nothing here launches a kernel)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ll_attn.h")


@pytest.fixture(scope="module")
def L():
    from log_linear_attention_chunked_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from log_linear_attention_chunked_gb300 import build
        build.build()
    return binding.lib()


def declared_symbols():
    inc = os.path.dirname(HEADER)
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    return sorted(set(re.findall(r"LL_API\s+[\w\s\*]+?\b(ll_\w+)\s*\(", src)))


def test_header_declares_the_abi():
    from log_linear_attention_chunked_gb300 import binding
    assert declared_symbols() == sorted(binding.SYMBOLS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    from log_linear_attention_chunked_gb300 import binding
    assert binding.ll_version() >= 100
    for code in range(7):
        assert binding.ll_status_str(code)
    assert binding.ll_status_str(99) == "unknown status"


def _shape(**kw):
    from log_linear_attention_chunked_gb300 import binding
    d = dict(B=1, H=2, T=64, dk=16, dv=16, L=7, chunk=16, Ls=0, io=binding.LL_F32)
    d.update(kw)
    return binding.make_shape(**d)


def test_workspace_size_queries(L):
    from log_linear_attention_chunked_gb300 import binding
    assert binding.ll_attn_fwd_workspace_size(_shape()) > 0
    assert binding.ll_attn_fwd_workspace_size(_shape(chunk=24)) == 0      # not a power of two
    assert binding.ll_attn_fwd_workspace_size(_shape(T=72, L=8)) > 0      # ragged T: partial last chunk
    assert binding.ll_gdn_fwd_workspace_size(_shape(T=72, L=8)) == 0       # Gated DeltaNet: whole chunks only
    assert binding.ll_attn_fwd_workspace_size(_shape(L=6)) == 0           # too few levels for T=64
    assert binding.ll_attn_fwd_workspace_size(_shape(dk=96)) == 0         # unsupported head dim
    big = binding.ll_attn_fwd_workspace_size(_shape(B=1, H=16, T=16384, dk=128, dv=128, L=15, chunk=64,
                                                    io=binding.LL_BF16))
    assert big > 0


FAKE = 0x7f0000000000  # never dereferenced: every case below fails a host-side check first


def _fwd(L, shape, ptrs=None, ws=FAKE, ws_bytes=1 << 40, state=None, scale=None):
    p = ptrs or [FAKE] * 6
    vp = ctypes.c_void_p
    return L.ll_attn_fwd(ctypes.byref(shape), *[vp(x) if x else None for x in p],
                         vp(state) if state else None, vp(scale) if scale else None,
                         vp(ws) if ws else None, ctypes.c_size_t(ws_bytes), None)


def test_fwd_rejects_bad_args_on_host(L):
    assert _fwd(L, _shape(chunk=24)) == 1
    assert _fwd(L, _shape(T=0)) == 1
    assert _fwd(L, _shape(dk=96)) == 2
    assert _fwd(L, _shape(), ptrs=[FAKE, 0, FAKE, FAKE, FAKE, FAKE]) == 1       # null k
    assert _fwd(L, _shape(), ptrs=[FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE]) == 1  # misaligned q
    assert _fwd(L, _shape(), ws=0) == 5                                         # no workspace
    assert _fwd(L, _shape(), ws_bytes=16) == 5                                  # workspace too small
    assert _fwd(L, _shape(), ws=FAKE + 16) == 5                                 # workspace not 256-aligned
    assert _fwd(L, _shape(Ls=7), state=FAKE) == 1                               # state without scale
    assert _fwd(L, _shape(Ls=6), state=FAKE, scale=FAKE) == 1                   # Ls < bit_length(T)


def test_decode_rejects_bad_args_on_host(L):
    vp = ctypes.c_void_p
    args = [vp(FAKE)] * 10
    assert L.ll_attn_decode_step(0, 1, 16, 16, 4, 0, *args) == 1
    assert L.ll_attn_decode_step(1, 1, 96, 16, 4, 0, *args) == 2
    assert L.ll_attn_decode_step(1, 1, 16, 16, 63, 0, *args) == 1
    bad = list(args)
    bad[3] = None
    assert L.ll_attn_decode_step(1, 1, 16, 16, 4, 0, *bad) == 1
    bad = list(args)
    bad[0] = vp(FAKE + 8)
    assert L.ll_attn_decode_step(1, 1, 16, 16, 4, 0, *bad) == 1


def test_cont_rejects_bad_args_on_host(L):
    from log_linear_attention_chunked_gb300 import binding
    vp = ctypes.c_void_p
    ok = _shape(T=64, L=12, Ls=10)                                       # t0 = 512: t1 = 576, bitlen 10
    assert L.ll_attn_fwd_cont_workspace_size(ctypes.byref(ok), 512) > 0
    # a start that is not a multiple of 64 runs as aligned pieces (96: 32, then 64 at 128, ...)
    assert L.ll_attn_fwd_cont_workspace_size(ctypes.byref(ok), 96) > 0
    assert L.ll_attn_fwd_cont_workspace_size(ctypes.byref(ok), -64) == 0
    assert L.ll_attn_fwd_cont_workspace_size(ctypes.byref(_shape(T=64, L=12, Ls=9)), 512) == 0  # slots
    assert L.ll_attn_fwd_cont_workspace_size(ctypes.byref(_shape(T=64, L=10, Ls=10)), 512) == 0  # levels
    args = [vp(FAKE)] * 10  # state_in, scale_in, q, k, v, log_alpha, lam, o, state_out, scale_out
    for i in range(8):      # every required tensor
        bad = list(args)
        bad[i] = None
        assert L.ll_attn_fwd_cont(ctypes.byref(ok), 512, *bad, vp(FAKE), ctypes.c_size_t(1 << 40), None) == 1, i
    bad = list(args)
    bad[9] = None           # state_out without scale_out
    assert L.ll_attn_fwd_cont(ctypes.byref(ok), 512, *bad, vp(FAKE), ctypes.c_size_t(1 << 40), None) == 1
    same = list(args)       # state_out overlapping state_in
    assert L.ll_attn_fwd_cont(ctypes.byref(ok), 512, *same, vp(FAKE), ctypes.c_size_t(1 << 40), None) == 1


def test_bwd_rejects_bad_args_on_host(L):
    from log_linear_attention_chunked_gb300 import binding
    vp = ctypes.c_void_p
    ok = _shape()
    assert binding.ll_attn_bwd_workspace_size(ok) > 0
    assert binding.ll_attn_bwd_workspace_size(_shape(T=72, L=8)) > 0     # ragged T
    assert binding.ll_attn_bwd_workspace_size(_shape(Ls=7)) == 0         # no state gradients
    assert binding.ll_attn_bwd_workspace_size(_shape(dk=96)) == 0
    assert binding.ll_attn_bwd_launches(ok) == 6

    def bwd(shape, ptrs, ws=FAKE, ws_bytes=1 << 40):
        return L.ll_attn_bwd(ctypes.byref(shape), *[vp(x) if x else None for x in ptrs],
                             vp(ws) if ws else None, ctypes.c_size_t(ws_bytes), None)

    # eleven tensors, each far from the others so that none overlap
    ptrs = [FAKE + (i << 32) for i in range(11)]
    assert bwd(_shape(Ls=7), ptrs) == 1
    assert bwd(_shape(dk=96), ptrs) == 2
    for i in range(11):     # every tensor is required
        bad = list(ptrs)
        bad[i] = 0
        assert bwd(ok, bad) == 1, i
    bad = list(ptrs)
    bad[6] = ptrs[0] + 16   # dq inside q
    assert bwd(ok, bad) == 1
    bad = list(ptrs)
    bad[10] = ptrs[7]       # dlam on dk
    assert bwd(ok, bad) == 1
    bad = list(ptrs)
    bad[2] = ptrs[2] + 8    # misaligned v
    assert bwd(ok, bad) == 1
    assert bwd(ok, ptrs, ws=0) == 5
    assert bwd(ok, ptrs, ws_bytes=16) == 5
    assert bwd(ok, ptrs, ws=FAKE + (20 << 32) + 16) == 5


def test_gdn_b_rejects_bad_args_on_host(L):
    vp = ctypes.c_void_p
    s = _shape(Ls=3)
    assert L.ll_gdn_fwd_b(ctypes.byref(s), *([vp(FAKE)] * 8), ctypes.c_size_t(1 << 40), None) == 1
    s = _shape()
    args = [vp(FAKE)] * 7
    for i in range(7):  # every null tensor
        bad = list(args)
        bad[i] = None
        assert L.ll_gdn_fwd_b(ctypes.byref(s), *bad, vp(FAKE), ctypes.c_size_t(1 << 40), None) == 1, i
    assert L.ll_gdn_fwd_b(ctypes.byref(s), *args, None, ctypes.c_size_t(0), None) in (2, 5)


def test_gdn_decode_rejects_bad_args_on_host(L):
    vp = ctypes.c_void_p
    args = [vp(FAKE)] * 10  # t, q, k, v, log_alpha, beta, lam, states, o, stream
    assert L.ll_gdn_decode_step(0, 1, 16, 16, 4, 0, *args) == 1            # B < 1
    assert L.ll_gdn_decode_step(1, 1, 96, 16, 4, 0, *args) == 2            # head dim
    assert L.ll_gdn_decode_step(1, 1, 16, 16, 63, 0, *args) == 1           # Ls > 62
    assert L.ll_gdn_decode_step(1, 1, 16, 16, 4, 5, *args) == 1            # io
    for i in range(9):                                                     # every null tensor
        bad = list(args)
        bad[i] = None
        assert L.ll_gdn_decode_step(1, 1, 16, 16, 4, 0, *bad) == 1, i
    bad = list(args)
    bad[5] = vp(FAKE + 4)                                                  # misaligned beta
    assert L.ll_gdn_decode_step(1, 1, 16, 16, 4, 0, *bad) == 1


def test_gdn_rejects_bad_args_on_host(L):
    from log_linear_attention_chunked_gb300 import binding
    vp = ctypes.c_void_p
    s = _shape(Ls=3)
    assert L.ll_gdn_fwd(ctypes.byref(s), *([vp(FAKE)] * 8), ctypes.c_size_t(1 << 40), None) == 1
    s = _shape()
    assert L.ll_gdn_fwd(ctypes.byref(s), *([vp(FAKE)] * 7), None, ctypes.c_size_t(0), None) in (2, 5)


def test_binding_fails_loudly_without_the_library(monkeypatch):
    """No fallback: a missing libllattn.so is an error, not a slower path."""
    from log_linear_attention_chunked_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", binding.LIB_PATH + ".absent")
    with pytest.raises(RuntimeError):
        binding.lib()


def test_product_path_does_not_reach_the_oracle():
    """The package and the benchmark's GPU arm never import the oracle: only the
    tests, smoke() and the benchmark's CPU-baseline and reference arms do."""
    import ast
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "log_linear_attention_chunked_gb300")
    for f in sorted(os.listdir(pkg)):
        if not f.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(pkg, f)).read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), (f, names)


def test_noalloc_scratch_size_matches_header():
    """The binding's copy of the no-allocation scratch size is the header's."""
    from log_linear_attention_chunked_gb300 import binding
    m = re.search(r"#define\s+LL_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(HEADER).read())
    assert m, "LL_NOALLOC_SCRATCH_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == binding.NOALLOC_SCRATCH_BYTES


def test_withhold_hook_rejects_bad_args_on_host(L):
    from log_linear_attention_chunked_gb300 import binding
    vp = ctypes.c_void_p
    s = binding.make_shape(1, 1, 256, 128, 128, 9, 64, 0, binding.LL_BF16)
    p = [vp(FAKE)] * 6
    # node out of range, limit out of range: refused before any launch
    assert L.ll_test_fwd_withhold_node(ctypes.byref(s), *p, vp(FAKE), 1 << 20, 2, 10 ** 6, None) == 1
    assert L.ll_test_fwd_withhold_node(ctypes.byref(s), *p, vp(FAKE), 1 << 20, 0, 10, None) == 1
    # a shape off the tensor-core path
    s2 = binding.make_shape(1, 1, 256, 32, 32, 9, 64, 0, binding.LL_BF16)
    assert L.ll_test_fwd_withhold_node(ctypes.byref(s2), *p, vp(FAKE), 1 << 20, 0, 10 ** 6, None) == 2
