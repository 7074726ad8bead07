"""The Python binding's marshalling, on the CPU.

The binding reads the C calls' sizes from tensor shapes and passes raw device
pointers, so it refuses host tensors and arguments whose shapes or element
types disagree before any call. Here the library is replaced by a recorder
(nothing runs), and the device check is relaxed where a test needs
consistent arguments to reach the recorder.
"""
import pytest
import torch

from paged_kv_cache_context_gb300 import pa


class Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(pa, "lib", lambda: rec)
    monkeypatch.setattr(pa, "_stream", lambda stream=None: 0)
    monkeypatch.setattr(pa, "_is_device_tensor", lambda t: True)
    return rec


def decode_args(S=3, Hq=8, Hkv=2, D=64, bs=16, NB=10, MB=4, qd=torch.bfloat16, cd=None):
    q = torch.zeros(S, Hq, D, dtype=qd)
    out = torch.zeros_like(q)
    k = torch.zeros(NB, Hkv, bs, D, dtype=cd or qd)
    bt = torch.zeros(S, MB, dtype=torch.int32)
    cl = torch.ones(S, dtype=torch.int32)
    return out, q, k, k.clone(), bt, cl


def test_host_tensors_are_refused_before_any_call(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(pa, "lib", lambda: rec)
    out, q, k, v, bt, cl = decode_args()
    with pytest.raises(ValueError, match="CUDA"):
        pa.decode(out, q, k, v, bt, cl, 2, 0.1)
    key = torch.zeros(5, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pa.reshape_and_cache(key, key, k, v, torch.zeros(5, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA"):
        pa.copy_blocks(k, v, torch.zeros(1, 2, dtype=torch.int32))
    assert rec.calls == []


def test_consistent_arguments_reach_the_c_call_with_their_sizes(fake):
    out, q, k, v, bt, cl = decode_args(S=3, Hq=8, Hkv=2, D=64, bs=16, NB=10, MB=4)
    pa.decode(out, q, k, v, bt, cl, 2, 0.125, window=0)
    name, args = fake.calls[-1]
    assert name == "pa_decode"
    assert args[6:13] == (3, 8, 2, 64, 16, 10, 4)  # S, Hq, Hkv, D, bs, NB, MB
    ks = torch.zeros(10, 2, 16, dtype=torch.float32)
    k8 = torch.zeros(10, 2, 16, 64, dtype=torch.int8)
    pa.decode_int8(out, q, k8, k8.clone(), ks, ks.clone(), bt, cl, 2, 0.125)
    assert fake.calls[-1][0] == "pa_decode_int8"
    key = torch.zeros(5, 2, 64, dtype=torch.bfloat16)
    pa.reshape_and_cache_int8(key, key, k8, k8.clone(), ks, ks.clone(),
                              torch.zeros(5, dtype=torch.int64))
    assert fake.calls[-1][1][7:12] == (5, 2, 64, 16, 10)  # T, Hkv, D, bs, NB
    qp = torch.zeros(7, 8, 64, dtype=torch.bfloat16)
    pa.prefill(torch.zeros_like(qp), qp, k, v, bt, torch.zeros(4, dtype=torch.int32), cl, 2, 5,
               0.125)
    assert fake.calls[-1][1][7:17] == (7, 3, 8, 2, 64, 16, 10, 4, 5, pytest.approx(0.125))


@pytest.mark.parametrize("bad", ["cache_dtype", "kv_heads", "head_dim", "out_shape", "out_dtype",
                                 "table_rows", "table_dtype", "lens", "v_shape"])
def test_decode_mismatches_raise(fake, bad):
    out, q, k, v, bt, cl = decode_args()
    kv_heads = 2
    if bad == "cache_dtype":
        k, v = k.float(), v.float()
    elif bad == "kv_heads":
        kv_heads = 4
    elif bad == "head_dim":
        q, out = torch.zeros(3, 8, 128, dtype=torch.bfloat16), torch.zeros(3, 8, 128,
                                                                           dtype=torch.bfloat16)
    elif bad == "out_shape":
        out = torch.zeros(3, 8, 32, dtype=torch.bfloat16)
    elif bad == "out_dtype":
        out = out.float()
    elif bad == "table_rows":
        bt = torch.zeros(4, 4, dtype=torch.int32)
    elif bad == "table_dtype":
        bt = bt.long()
    elif bad == "lens":
        cl = torch.ones(2, dtype=torch.int32)
    elif bad == "v_shape":
        v = torch.zeros(9, 2, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.decode(out, q, k, v, bt, cl, kv_heads, 0.1)
    assert fake.calls == []


def test_write_and_int8_mismatches_raise(fake):
    _, _, k, v, _, _ = decode_args()
    key = torch.zeros(5, 2, 64, dtype=torch.bfloat16)
    sm = torch.zeros(5, dtype=torch.int64)
    with pytest.raises(ValueError):  # FP8 caches are bytes
        pa.reshape_and_cache(key, key, k, v, sm, "fp8_e4m3", 1.0, 1.0)
    with pytest.raises(ValueError):  # one slot per token
        pa.reshape_and_cache(key, key, k, v, sm[:4])
    with pytest.raises(ValueError):
        pa.reshape_and_cache(key, key, k, v, sm.int())
    k8 = torch.zeros(10, 2, 16, 64, dtype=torch.int8)
    with pytest.raises(ValueError):  # one scale per cached row
        pa.reshape_and_cache_int8(key, key, k8, k8.clone(), torch.zeros(10, 2, dtype=torch.float32),
                                  torch.zeros(10, 2, dtype=torch.float32), sm)
    with pytest.raises(ValueError):
        pa.copy_blocks(k, v, torch.zeros(3, dtype=torch.int32))
    assert fake.calls == []
