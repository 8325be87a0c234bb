"""ll_attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers can neither pass a workspace nor allocate one (a host runtime
that owns all device memory after start-up, a plugin without an allocator, a
loop that must not risk a synchronising cudaMalloc).  The no-allocation entry
point runs the same forward with the library's own fixed scratch array; this
test calls it through the C ABI and checks it against ll_attn_fwd, twice in a
row with different inputs, so a second call cannot pass on the first call's
leftovers.  The cases cover both forward paths: the CUDA-core kernels (float32
d=16, bf16 d=64) and the tensor-core kernel (bf16 d=128), whose per-call
publication words in the scratch are the part a stale array could confuse;
the tensor-core case also exports the decode states.  The file sorts last so
a failure here never hides another test.
"""

import ctypes

import pytest
import torch

from oracle.partition import levels_needed
from log_linear_attention_chunked_gb300 import synth
from tests._parity import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from log_linear_attention_chunked_gb300 import binding
    binding.lib()
    return binding


def _inputs(io, T, d, H, tag):
    cfg = dict(synth.WORKLOADS["mamba2_fp32_t64"], io=io, T=T, dk=d, dv=d, L=levels_needed(T), B=1, H=H)
    dev = torch.device("cuda")
    return {n: x.to(dev) for n, x in synth.make_inputs(cfg, tag=tag).items()}, cfg


@pytest.mark.parametrize("io,T,d,H,chunk,Ls", [("f32", 64, 16, 2, 16, 0), ("bf16", 1024, 64, 4, 64, 0),
                                               ("bf16", 1024, 128, 2, 64, 0), ("bf16", 1280, 128, 2, 64, 12)])
def test_noalloc_matches_workspace_entry_point(B, io, T, d, H, chunk, Ls):
    tol = TOL_F32 if io == "f32" else TOL_BF16
    for call in range(2):
        g, cfg = _inputs(io, T, d, H, tag=f"noalloc{call}")
        shape = B.make_shape(1, H, T, d, d, cfg["L"], chunk, Ls, B._io(g["q"].dtype))
        assert B.ll_attn_fwd_workspace_size(shape) <= B.NOALLOC_SCRATCH_BYTES
        if d == 128:
            assert B.ll_attn_fwd_launches(shape) == (2 if Ls else 1), "tensor-core path not selected"
        st_ref = sc_ref = st = sc = None
        if Ls:
            st_ref = torch.empty(1, H, Ls, d, d, device="cuda")
            sc_ref = torch.empty(1, H, Ls, device="cuda")
            st = torch.full_like(st_ref, float("nan"))
            sc = torch.full_like(sc_ref, float("nan"))
        ref = B.ll_attn_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], chunk, state_out=st_ref,
                            scale_out=sc_ref)
        o = torch.full_like(ref, float("nan"))
        B.ll_attn_fwd_noalloc(g["q"], g["k"], g["v"], g["log_alpha"], g["lam"], chunk, o=o, state_out=st,
                              scale_out=sc)
        assert B.ll_last_device_error() == 0
        assert torch.isfinite(o.float()).all()
        assert rel_err(o.float().cpu().numpy(), ref.float().cpu().numpy()) <= tol, call
        if Ls:
            assert torch.equal(sc, sc_ref), call
            assert rel_err(st.cpu().numpy(), st_ref.cpu().numpy()) <= tol, call


def test_noalloc_rejects_shapes_beyond_the_scratch(B):
    # a workload whose workspace exceeds the fixed scratch is refused on the
    # host; the data pointers are null, so a regression that reached the
    # forward would stop at its null-pointer check instead of launching
    shape = B.make_shape(1, 16, 16384, 128, 128, 15, 64, 0, B.LL_BF16)
    assert B.ll_attn_fwd_workspace_size(shape) > B.NOALLOC_SCRATCH_BYTES
    st = B.lib().ll_attn_fwd_noalloc(ctypes.byref(shape), *[None] * 9)
    assert st == 5  # LL_ERR_WORKSPACE
