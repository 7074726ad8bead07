"""The five named workloads at full size, in the launch configuration the
benchmark times (pa_decode with the split plan's workspace): sampled
(sequence, head) rows against the oracle, the cache bytes of the sampled
sequences bit for bit, and properties of the whole output (finite, no device
error). Values are drawn on the GPU with a seeded CUDA generator; the oracle
gets host copies of exactly those rows.
"""
import pytest
import torch

import oracle
from _gpu import DEV, assert_close, bits, device_errors, gpu_caches, gpu_decode
from _helpers import oracle_caches_for, sampled_seqs
from paged_kv_cache_context_gb300 import build, pa
from paged_kv_cache_context_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pa.lib()
    device_errors()


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_full_size_workload_sampled(name):
    case = wl.config(name, value_device=DEV)
    kg, vg = gpu_caches(case)
    out = gpu_decode(case, kg, vg, split=True)
    torch.cuda.synchronize()
    assert device_errors() == 0
    assert torch.isfinite(out.float()).all()

    seqs = sampled_seqs(case)
    ko, vo = oracle_caches_for(case, seqs)
    # the sampled sequences' blocks are bit-identical
    blocks = torch.unique(case.block_tables[seqs].flatten())
    blocks = blocks[blocks >= 0].long()
    assert torch.equal(bits(kg[blocks.to(DEV)]), bits(ko[blocks]))
    assert torch.equal(bits(vg[blocks.to(DEV)]), bits(vo[blocks]))
    rows = [s * case.num_heads + h for s in seqs for h in range(case.num_heads)]
    ref = oracle.decode(case.query, ko, vo, case.block_tables, case.context_lens,
                        case.num_kv_heads, case.block_size, case.scale, case.window,
                        case.kv_dtype, case.k_scale, case.v_scale, rows=rows)
    assert_close(case, out, ref, rows=rows, what=name)
