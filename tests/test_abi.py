"""The C ABI without a GPU: the library loads, exports every entry point that
include/pa.h declares, and rejects bad arguments on the host with the
documented status codes before touching the device (fake non-NULL pointers
are never dereferenced on these paths)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_context_gb300 import build, pa
    build.build()
    return pa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(pa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pa_reshape_and_cache", "pa_decode", "pa_reduce", "pa_slot_mapping",
                 "pa_decode_partials", "pa_decode_plan", "pa_decode_workspace_size",
                 "pa_decode_cascade", "pa_decode_cascade_workspace_size", "pa_copy_blocks",
                 "pa_block_budget", "pa_reshape_and_cache_int8", "pa_decode_int8",
                 "pa_prefill", "pa_prefill_int8", "pa_prefill_fp8", "pa_decode_cascade_fp8",
                 "pa_decode_cascade_int8",
                 "pa_get_device_error", "pa_status_string", "pa_version"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    from paged_kv_cache_context_gb300 import pa
    for code in range(0, -12, -1):
        assert pa.status_string(code) and pa.status_string(code) != "unknown status"
    assert pa.status_string(-99) == "unknown status"
    assert pa.version() >> 16 == 1


P = 4096  # a fake, 16-byte aligned, never-dereferenced pointer


def decode_call(L, **kw):
    a = dict(out=P, query=P, k=P, v=P, bt=P, cl=P, S=2, Hq=8, Hkv=2, D=128, bs=32, NB=10, MB=4,
             scale=0.1, window=0, qd=1, kvd=0, ks=1.0, vs=1.0, ws=None, wsb=0)
    a.update(kw)
    return L.pa_decode(a["out"], a["query"], a["k"], a["v"], a["bt"], a["cl"], a["S"], a["Hq"],
                       a["Hkv"], a["D"], a["bs"], a["NB"], a["MB"], a["scale"], a["window"],
                       a["qd"], a["kvd"], a["ks"], a["vs"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(query=None), -1), (dict(bt=None), -1), (dict(cl=None), -1),
    (dict(qd=7), -2), (dict(kvd=5), -2),
    (dict(Hq=7), -3), (dict(Hq=18, Hkv=2), -3), (dict(S=-1), -3), (dict(NB=0), -3),
    (dict(MB=0), -3), (dict(S=70000), -3),
    (dict(D=80), -4), (dict(D=256), -4),
    (dict(bs=8), -5), (dict(bs=128), -5),
    (dict(window=-32), -6), (dict(window=48), -6), (dict(window=32 * 5), -6),
    (dict(kvd=1, ks=0.0), -11), (dict(kvd=1, vs=float("inf")), -11),
    (dict(kvd=1, ks=float("nan")), -11),
    (dict(query=P + 8), -10), (dict(k=P + 2), -10),
])
def test_decode_rejects_bad_arguments_on_host(L, kw, code):
    assert decode_call(L, **kw) == code


def test_decode_empty_batch_is_a_noop(L):
    assert decode_call(L, S=0, query=None, out=None) == 0


def test_write_rejects_bad_arguments_on_host(L):
    f = L.pa_reshape_and_cache
    ok = dict(key=P, value=P, k=P, v=P, sm=P, T=4, H=2, D=64, bs=32, NB=8, ind=1, kvd=0,
              ks=1.0, vs=1.0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["key"], a["value"], a["k"], a["v"], a["sm"], a["T"], a["H"], a["D"], a["bs"],
                 a["NB"], a["ind"], a["kvd"], a["ks"], a["vs"], None)

    assert call(T=0, key=None) == 0
    assert call(key=None) == -1 and call(sm=None) == -1
    assert call(ind=9) == -2 and call(kvd=3) == -2
    assert call(T=-1) == -3 and call(H=0) == -3 and call(NB=0) == -3
    assert call(D=60) == -4 and call(bs=0) == -5
    assert call(kvd=1, ks=-1.0) == -11
    assert call(k=P + 4) == -10


def test_reduce_and_slot_mapping_reject_bad_arguments(L):
    assert L.pa_reduce(P, P, P, P, 0, 4, 64, 2, 1, None) == 0
    assert L.pa_reduce(P, None, P, P, 2, 4, 64, 2, 1, None) == -1
    assert L.pa_reduce(P, P, P, P, 2, 4, 63, 2, 1, None) == -4
    assert L.pa_reduce(P, P, P, P, 2, 4, 64, 0, 1, None) == -3
    assert L.pa_reduce(P, P + 4, P, P, 2, 4, 64, 2, 1, None) == -10
    assert L.pa_slot_mapping(P, P, None, P, 0, 1, 1, 32, 0, None) == 0
    assert L.pa_slot_mapping(P, None, None, P, 3, 1, 1, 32, 0, None) == -1
    assert L.pa_slot_mapping(P, P, None, P, 3, 1, 1, 32, 40, None) == -6


def test_split_plan_is_host_only_and_covers_the_context():
    from paged_kv_cache_context_gb300 import pa
    for S, Hkv, MB, W in [(32, 8, 128, 0), (8, 8, 128, 4096), (64, 32, 256, 0),
                          (128, 8, 81, 0), (2, 4, 2, 0), (1, 1, 4096, 0)]:
        ns, pps = pa.decode_plan(S, 4 * Hkv if Hkv < 32 else Hkv, Hkv, 128, 32, MB, W)
        pages = W // 32 if W else MB
        assert ns >= 1 and pps >= 1 and ns * pps >= pages
        assert (ns - 1) * pps < pages  # no split is entirely past the table


def test_balanced_workspace_depends_only_on_group_and_head_dim():
    """An arrival counter per persistent CTA (3840 bytes for 152 x 6 CTAs), then
    two partial slots of G' x D floats (G' = group rounded up to 1, 2, 4 or 8)
    plus their (max, sum) per CTA."""
    from paged_kv_cache_context_gb300 import pa
    for Hq, Hkv, D, gt in [(32, 8, 128, 4), (32, 32, 96, 1), (12, 4, 64, 4), (56, 8, 128, 8)]:
        sizes = {pa.decode_workspace_size(S, Hq, Hkv, D, 32, MB, 0)
                 for S, MB in [(1, 1), (32, 128), (4096, 4096)]}
        assert len(sizes) == 1
        ws = sizes.pop()
        slots = 152 * 6 * 2
        assert ws >= 3840 + slots * (gt * D * 4 + gt * 2 * 4)
        assert ws <= 3840 + slots * (gt * D * 4 + gt * 2 * 4) + 2 * 256
    assert pa.decode_workspace_size(2, 6, 4, 128, 32, 8, 0) == 0  # 6 % 4 != 0
    assert pa.decode_workspace_size(2, 32, 4, 128, 32, 8, 0) <= 8 << 20  # G = 8, D = 128


def test_balanced_entry_points_reject_bad_arguments_on_host(L):
    n = ctypes.c_int(7)
    args = [P, P, P, P, P, P, 2, 8, 2, 128, 32, 10, 4, 0.1, 0, 1, 0, 1.0, 1.0]
    assert L.pa_decode_balanced(*args, None, 0, ctypes.addressof(n), None) == -1
    assert n.value == 0
    assert L.pa_decode_balanced(*args, P, 1024, ctypes.addressof(n), None) == -7
    assert L.pa_decode_balanced(*args, P, 1 << 30, None, None) == -1
    assert L.pa_decode_workspace_clear(None, 4096, None) == -1
    assert L.pa_decode_workspace_clear(P, 2559, None) == -7
    assert L.pa_decode_workspace_clear(P + 4, 4096, None) == -10


def test_cascade_and_copy_blocks_reject_bad_arguments_on_host(L):
    from paged_kv_cache_context_gb300 import pa
    ws = pa.decode_cascade_workspace_size(4, 8, 2, 128, 32, 3)
    assert ws > 0 and pa.decode_cascade_workspace_size(8, 8, 2, 128, 32, 3) > ws
    assert pa.decode_cascade_workspace_size(4, 6, 4, 128, 32, 3) == 0

    def call(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, cl=P, S=4, Hq=8, Hkv=2, D=128, bs=32, NB=40, MB=8,
                 scale=0.1, qd=1, pp=3, ws=P, wsb=1 << 30)
        a.update(kw)
        return L.pa_decode_cascade(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["S"],
                                   a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"], a["MB"],
                                   a["scale"], a["qd"], a["pp"], a["ws"], a["wsb"], None)

    assert call(S=0, q=None) == 0
    assert call(ws=None) == -1 and call(bt=None) == -1
    assert call(qd=0) == -2                     # fp32 queries: no tensor-core prefix path
    assert call(D=96) == -4
    assert call(pp=0) == -3 and call(pp=9) == -3
    assert call(wsb=1024) == -7
    assert call(ws=P + 4) == -10

    # the 8-bit caches: the same checks, with the FP8 scales and INT8 row scales
    def fp8(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, cl=P, S=4, Hq=8, Hkv=2, D=128, bs=32, NB=40, MB=8,
                 scale=0.1, ks=1.0, vs=1.0, qd=1, pp=3, ws=P, wsb=1 << 30)
        a.update(kw)
        return L.pa_decode_cascade_fp8(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"],
                                       a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
                                       a["MB"], a["scale"], a["ks"], a["vs"], a["qd"], a["pp"],
                                       a["ws"], a["wsb"], None)

    assert fp8(S=0, q=None) == 0
    assert fp8(ws=None) == -1 and fp8(qd=0) == -2 and fp8(D=96) == -4 and fp8(pp=9) == -3
    assert fp8(ks=0.0) == -11 and fp8(vs=float("nan")) == -11
    assert fp8(wsb=1024) == -7

    def int8(**kw):
        a = dict(out=P, q=P, k=P, v=P, ksc=P, vsc=P, bt=P, cl=P, S=4, Hq=8, Hkv=2, D=64, bs=16,
                 NB=40, MB=8, scale=0.1, qd=2, pp=3, ws=P, wsb=1 << 30)
        a.update(kw)
        return L.pa_decode_cascade_int8(a["out"], a["q"], a["k"], a["v"], a["ksc"], a["vsc"],
                                        a["bt"], a["cl"], a["S"], a["Hq"], a["Hkv"], a["D"],
                                        a["bs"], a["NB"], a["MB"], a["scale"], a["qd"], a["pp"],
                                        a["ws"], a["wsb"], None)

    assert int8(S=0, q=None) == 0
    assert int8(ksc=None) == -1 and int8(ws=None) == -1
    assert int8(qd=0) == -2 and int8(D=96) == -4 and int8(pp=0) == -3
    assert int8(ksc=P + 4) == -10 and int8(wsb=64) == -7
    f = L.pa_copy_blocks
    assert f(P, P, P, 0, 2, 64, 32, 10, 2, None) == 0
    assert f(P, None, P, 1, 2, 64, 32, 10, 2, None) == -1
    assert f(P, P, P, 1, 2, 64, 32, 10, 3, None) == -2
    assert f(P, P, P, 1, 1, 4, 1, 10, 1, None) == -4   # 4-byte blocks
    assert f(P, P, P, -1, 2, 64, 32, 10, 2, None) == -3
    assert f(P + 8, P, P, 1, 2, 64, 32, 10, 2, None) == -10


def test_block_budget_closed_forms(L):
    """Pool sizing by a memory amount in MB, a fraction of memory, or a context
    size ("PagedAttention in mistral.rs", Using the CLI and the Rust API): one
    block is block_size tokens of K and V for every kv head of every layer."""
    import torch
    from paged_kv_cache_context_gb300 import pa
    bf, f32 = torch.bfloat16, torch.float32
    # 32 layers x K,V x 8 kv heads x 32 tokens x 128 dims x 2 bytes = 4 MiB a block
    assert pa.block_budget(32, 8, 128, 32, bf, mb=4096) == 1024
    assert pa.block_budget(32, 8, 128, 32, bf, mb=4095.99) == 1023
    assert pa.block_budget(32, 8, 128, 32, bf, mb=3.99) == 0
    # an FP8 cache holds twice the blocks of a 16-bit one, fp32 half
    for mb in (1, 100, 777.5, 40_000):
        n16 = pa.block_budget(4, 2, 64, 16, bf, mb=mb)
        assert pa.block_budget(4, 2, 64, 16, bf, "fp8_e4m3", mb=mb) in (2 * n16, 2 * n16 + 1)
        assert pa.block_budget(4, 2, 64, 16, f32, mb=mb) == n16 // 2
        # the FP8 cache's size does not depend on the query type
        assert (pa.block_budget(4, 2, 64, 16, f32, "fp8_e4m3", mb=mb)
                == pa.block_budget(4, 2, 64, 16, bf, "fp8_e4m3", mb=mb))
    # 0.95 of memory, the CLI's example fraction
    blk = 32 * 2 * 8 * 32 * 128 * 2
    assert pa.block_budget(32, 8, 128, 32, bf, fraction=1.0, available_bytes=100 * blk) == 100
    assert pa.block_budget(32, 8, 128, 32, bf, fraction=0.95, available_bytes=100 * blk) == 95
    assert pa.block_budget(32, 8, 128, 32, bf, fraction=0.95, available_bytes=100 * blk - 1) == 94
    # a 1024-token context in 32-token blocks, the Rust API's example
    assert pa.block_budget(32, 8, 128, 32, bf, context_tokens=1024) == 32
    assert pa.block_budget(32, 8, 128, 32, bf, context_tokens=1025) == 33
    assert pa.block_budget(32, 8, 128, 32, bf, context_tokens=0) == 0
    # rejected on the host
    f = L.pa_block_budget
    assert f(0, 1.0, 0, 0, 8, 128, 32, 1, 0) == -3
    assert f(0, 1.0, 0, 32, 0, 128, 32, 1, 0) == -3
    assert f(0, 1.0, 0, 32, 8, 0, 32, 1, 0) == -4
    assert f(0, 1.0, 0, 32, 8, 128, 0, 1, 0) == -3
    assert f(0, 1.0, 0, 32, 8, 128, 32, 5, 0) == -2
    assert f(0, 1.0, 0, 32, 8, 128, 32, 1, 3) == -2
    assert f(0, -1.0, 0, 32, 8, 128, 32, 1, 0) == -3
    assert f(0, float("nan"), 0, 32, 8, 128, 32, 1, 0) == -3
    assert f(1, 1.5, 1 << 30, 32, 8, 128, 32, 1, 0) == -3
    assert f(3, 1.0, 0, 32, 8, 128, 32, 1, 0) == -3
    with pytest.raises(ValueError):
        pa.block_budget(32, 8, 128, 32, bf, mb=1, context_tokens=1)
    # an INT8 row is D bytes plus its 4-byte scale: 32*2*8*32*(128+4) bytes a block
    assert pa.block_budget(32, 8, 128, 32, bf, "int8", mb=4096) == (4096 << 20) // (
        32 * 2 * 8 * 32 * 132)
    assert pa.block_budget(1, 1, 64, 16, bf, "int8", mb=2 * 16 * 68 / 2 ** 20 * 5) == 5


def test_int8_entry_points_reject_bad_arguments_on_host(L):
    d = L.pa_decode_int8

    def dec(**kw):
        a = dict(out=P, q=P, k=P, v=P, ks=P, vs=P, bt=P, cl=P, S=4, Hq=8, Hkv=2, D=128, bs=32,
                 NB=10, MB=8, scale=0.1, W=0, qd=1, ws=None, wsb=0)
        a.update(kw)
        return d(a["out"], a["q"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["cl"], a["S"],
                 a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"], a["MB"], a["scale"], a["W"],
                 a["qd"], a["ws"], a["wsb"], None)

    assert dec(S=0, q=None) == 0
    assert dec(ks=None) == -1 and dec(vs=None) == -1 and dec(k=None) == -1
    assert dec(qd=0) == -2 and dec(qd=7) == -2        # fp32 queries are not built for INT8
    assert dec(D=80) == -4 and dec(bs=8) == -5 and dec(Hq=7) == -3
    assert dec(W=48) == -6
    assert dec(ks=P + 4) == -10 and dec(vs=P + 8) == -10
    w = L.pa_reshape_and_cache_int8
    assert w(P, P, P, P, P, P, P, 0, 2, 128, 32, 10, 1, None) == 0
    assert w(P, P, P, P, None, P, P, 4, 2, 128, 32, 10, 1, None) == -1
    assert w(P, P, P, P, P, P, P, 4, 2, 128, 32, 10, 5, None) == -2
    assert w(P, P, P, P, P, P, P, 4, 2, 264, 32, 10, 1, None) == -4
    assert w(P, P, P, P, P, P, P, 4, 2, 100, 32, 10, 1, None) == -4
    assert w(P, P, P, P, P, P, P, 4, 2, 128, 0, 10, 1, None) == -5
    assert w(P, P, P, P, P, P, P, -1, 2, 128, 32, 10, 1, None) == -3
    assert w(P, P, P, P, P + 4, P, P, 4, 2, 128, 32, 10, 1, None) == -10
    # the native-cache entry points take no row scales, so they refuse INT8
    assert L.pa_decode(P, P, P, P, P, P, 4, 8, 2, 128, 32, 10, 8, 0.1, 0, 1, 2, 1.0, 1.0, None,
                       0, None) == -2
    assert L.pa_reshape_and_cache(P, P, P, P, P, 4, 2, 128, 32, 10, 1, 2, 1.0, 1.0, None) == -2


def test_prefill_rejects_bad_arguments_on_host(L):
    f = L.pa_prefill

    def call(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, cu=P, cl=P, T=40, S=4, Hq=8, Hkv=2, D=128, bs=32,
                 NB=10, MB=8, mq=16, scale=0.1, qd=1)
        a.update(kw)
        return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cu"], a["cl"], a["T"], a["S"],
                 a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"], a["MB"], a["mq"], a["scale"],
                 a["qd"], None)

    assert call(T=0, q=None) == 0 and call(S=0, q=None) == 0
    assert call(T=-1) == -3 and call(S=70000) == -3
    assert call(cu=None) == -1 and call(cl=None) == -1 and call(bt=None) == -1
    assert call(qd=0) == -2 and call(qd=4) == -2
    assert call(Hq=6, Hkv=4) == -3 and call(Hq=32, Hkv=2) == -3
    assert call(D=96) == -4 and call(bs=8) == -5
    assert call(mq=0) == -3 and call(mq=41) == -3
    assert call(out=P + 2) == -10 and call(k=P + 8) == -10


def test_8bit_prefill_rejects_bad_arguments_on_host(L):
    """pa_prefill_fp8 and pa_prefill_int8 share pa_prefill's checks, plus the
    FP8 scales (finite, positive) and the INT8 row scales (present, aligned)."""
    def fp8(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, cu=P, cl=P, T=40, S=4, Hq=8, Hkv=2, D=128, bs=32,
                 NB=10, MB=8, mq=16, scale=0.1, ks=0.5, vs=2.0, qd=1)
        a.update(kw)
        return L.pa_prefill_fp8(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cu"], a["cl"],
                                a["T"], a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
                                a["MB"], a["mq"], a["scale"], a["ks"], a["vs"], a["qd"], None)

    assert fp8(T=0, q=None) == 0
    assert fp8(cu=None) == -1 and fp8(qd=0) == -2 and fp8(D=96) == -4 and fp8(bs=8) == -5
    assert fp8(ks=0.0) == -11 and fp8(vs=-1.0) == -11 and fp8(ks=float("inf")) == -11
    assert fp8(ks=float("nan")) == -11
    assert fp8(k=P + 8) == -10

    def int8(**kw):
        a = dict(out=P, q=P, k=P, v=P, ksc=P, vsc=P, bt=P, cu=P, cl=P, T=40, S=4, Hq=8, Hkv=2,
                 D=64, bs=16, NB=10, MB=8, mq=16, scale=0.1, qd=2)
        a.update(kw)
        return L.pa_prefill_int8(a["out"], a["q"], a["k"], a["v"], a["ksc"], a["vsc"], a["bt"],
                                 a["cu"], a["cl"], a["T"], a["S"], a["Hq"], a["Hkv"], a["D"],
                                 a["bs"], a["NB"], a["MB"], a["mq"], a["scale"], a["qd"], None)

    assert int8(S=0, q=None) == 0
    assert int8(ksc=None) == -1 and int8(vsc=None) == -1
    assert int8(qd=0) == -2 and int8(D=96) == -4
    assert int8(vsc=P + 4) == -10


def test_int8_widening_identity_holds_for_every_code():
    """The decode widens INT8 codes without a conversion instruction: with the
    code's sign bit flipped, u = c + 128 is placed as the low byte of the
    binary32 bit pattern 0x4B0000uu (= 2^23 + u), and 2^23 + 128 is
    subtracted. Restated here in numpy for all 256 codes: the result is c,
    exactly."""
    import numpy as np
    c = np.arange(-128, 128, dtype=np.int32)
    u = (c.astype(np.uint32) & 0xFF) ^ 0x80
    f = (np.uint32(0x4B000000) | u).view(np.float32)
    assert np.array_equal(f - np.float32(8388736.0), c.astype(np.float32))
