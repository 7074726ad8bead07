"""pa_decode_static_scratch: paged decode for callers that cannot allocate.

Callers that have no allocator to hand pa_decode a workspace (a host program
that owns all device memory, or code that must never call cudaMalloc) use this
entry point; it keeps the split partials in the library's own fixed device
array. These tests call it through the C ABI and check that two calls in a
row (different shapes, so the second starts from what the first left in the
shared array) match the oracle's decode, and what pa_decode gives, within the
decode tolerance, and that a plan too large for the array is refused without
launching anything.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

STATIC_SCRATCH_BYTES = 8 << 20


def _fn():
    build.build()
    f = pa.lib().pa_decode_static_scratch
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, F, F, P]
    f.restype = I
    return f


def call_static(f, out, q, kc, vc, bt, cl, case, stream):
    S, Hq, D = q.shape
    NB, _, bs, _ = kc.shape
    return f(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
             cl.data_ptr(), S, Hq, case.num_kv_heads, D, bs, NB, bt.shape[1], case.scale,
             case.window, pa._DTYPE[case.q_dtype], pa._KV[case.kv_dtype], case.k_scale,
             case.v_scale, stream)


@pytest.mark.gpu
def test_static_scratch_matches_oracle_and_pa_decode_on_two_calls_in_a_row():
    from _gpu import DEV, assert_close, device_errors, gpu_caches, gpu_decode, to_dev
    from _helpers import oracle_caches, oracle_decode
    f = _fn()
    stream = torch.cuda.current_stream().cuda_stream
    device_errors()
    cases = [wl.scaled_config("mistral_bf16", 6, 8), wl.scaled_config("fp8_phi3", 6, 8)]
    prepared = []
    for case in cases:
        need = pa.decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                        case.head_dim, case.block_size,
                                        case.max_blocks_per_seq, case.window)
        assert 0 < need <= STATIC_SCRATCH_BYTES  # the split path really runs
        kc, vc = gpu_caches(case)
        ko, vo = oracle_caches(case)
        ref = oracle_decode(case, ko, vo)
        dec = gpu_decode(case, kc, vc, split=True).float().cpu()
        prepared.append((case, kc, vc, ref, dec))
    for case, kc, vc, ref, dec in prepared:  # two calls in a row through the C ABI
        out = torch.full(case.query.shape, float("nan"), dtype=case.q_dtype, device=DEV)
        rc = call_static(f, out, to_dev(case.query), kc, vc, to_dev(case.block_tables),
                         to_dev(case.context_lens), case, stream)
        assert rc == 0, pa.status_string(rc)
        assert_close(case, out, ref, what=f"static scratch vs oracle, {case.name}")
        assert_close(case, out, dec.double().numpy(), what=f"static scratch vs pa_decode, "
                                                          f"{case.name}")
    assert device_errors() == 0


def test_static_scratch_refuses_sizes_beyond_its_array():
    """Partial storage grows with the head dimension: head_dim 2048 with 8
    query heads per kv head would need ~80 MB, more than the fixed array, so
    the call is refused with PA_ERR_WORKSPACE before anything is enqueued (the
    pointers below are never dereferenced). Every supported shape fits."""
    f = _fn()
    need = pa.decode_workspace_size(4, 64, 8, 2048, 32, 16, 0)
    assert need > STATIC_SCRATCH_BYTES
    for Hq, Hkv, D in [(64, 8, 128), (32, 32, 96), (16, 16, 64)]:
        assert pa.decode_workspace_size(4, Hq, Hkv, D, 32, 16, 0) <= STATIC_SCRATCH_BYTES
    P = 4096
    rc = f(P, P, P, P, P, P, 4, 64, 8, 2048, 32, 100, 16, 0.1, 0, pa.PA_BF16, 0, 1.0, 1.0, None)
    assert rc == -7 and "workspace" in pa.status_string(rc)
