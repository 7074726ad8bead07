"""The bounded waits of the decode kernel give up instead of hanging.

With the library's test hook every CTA's producer stops before arming one of
its stages, so no copy is ever issued for it: the consumer warps' bounded wait
for that stage runs out, the kernel sets PA_DEVERR_TIMEOUT and every CTA ends
in order (it waits for the copies it did issue). The host reads the error bit,
and the context stays usable: the next decode, with the hook off, matches the
oracle.
"""
import pytest
import torch

from _gpu import DEV, assert_close, device_errors, gpu_caches, gpu_decode
from _helpers import oracle_caches, oracle_decode
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split", [True, False])
def test_wait_for_an_unarmed_stage_times_out_and_the_context_survives(split):
    build.build()
    pa.lib()
    device_errors()
    case = wl.scaled_config("mistral_bf16", 6, 8)
    kg, vg = gpu_caches(case)
    torch.cuda.synchronize()
    assert device_errors() == 0
    try:
        pa.test_set_unarmed_page(0)  # no CTA arms a single stage: nothing is in flight
        gpu_decode(case, kg, vg, split=split)
        torch.cuda.synchronize()
    finally:
        pa.test_set_unarmed_page(-1)
    assert device_errors() & 8  # PA_DEVERR_TIMEOUT
    ko, vo = oracle_caches(case)
    out = gpu_decode(case, kg, vg, split=split)
    assert_close(case, out, oracle_decode(case, ko, vo), what="decode after a timed-out launch")
    assert device_errors() == 0
