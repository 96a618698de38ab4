"""The C-ABI library builds, loads and exports every entry point the header declares;
host-only entry points validate configurations (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    from residual_kv_cache_gb300 import build
    return build.build()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "rkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rkv_[a-z_]+)\s*\(", text)))


def test_header_functions_are_exported(built):
    import residual_kv_cache_gb300 as rkv
    names = _header_functions()
    assert len(names) >= 12
    handle = ctypes.CDLL(built)
    for n in names:
        assert hasattr(handle, n), f"{n} missing from librkv.so"
    assert set(names) == set(rkv.ABI_FUNCTIONS), "binding and header disagree"


def test_library_has_sm103a_code(built):
    data = open(built, "rb").read()
    assert b"sm_103a" in data or b"sm_103" in data


def test_storage_bytes_and_config_validation(built):
    import residual_kv_cache_gb300 as rkv
    cfg = rkv.Config(n_kv_heads=8, head_dim=128, d_c=512, d_ff=1536, bits=4, ref_stride=16,
                     max_tokens=32768)
    s = rkv.storage_bytes(cfg)
    assert len(s) == 6 and s[0] == 2048 * 2048 and s[1] == 2048 * 4 and s[2] == 2048 * 4
    assert s[3] == 32768 * 256 and s[4] == 32768 * 16 * 4 and s[5] == 32768 * 4 * 4
    for bad in (dict(head_dim=96), dict(d_c=100), dict(d_c=576), dict(bits=3), dict(topk=5), dict(d_ff=200),
                dict(group=16), dict(max_refs=10), dict(ref_alpha=-0.1), dict(ref_sink=-1),
                dict(ref_alpha=float("nan")), dict(ref_alpha=0.02, ref_sink=4, max_refs=100)):
        with pytest.raises(rkv.RkvError) as e:
            rkv.storage_bytes(rkv.Config(**{**cfg.__dict__, **bad}))
        assert e.value.status == -1


def test_pool_size_follows_the_reference_schedule(built):
    """max_refs = 0 sizes the pool to the schedule's positions below max_tokens
    (ResidualKV notes §2.6), the count the oracle's schedule gives."""
    import residual_kv_cache_gb300 as rkv
    from oracle import codec as C
    for T, s, alpha, sink in ((32768, 16, 0.0, 0), (1000, 10, 0.0, 0), (262144, 10, 0.02, 0),
                              (262144, 10, 0.001, 4), (4096, 16, 0.02, 4), (300, 8, 5.0, 16)):
        cfg = rkv.Config(n_kv_heads=8, head_dim=128, d_c=512, d_ff=1536, ref_stride=s,
                         max_tokens=T, ref_alpha=alpha, ref_sink=sink)
        R = len(C.reference_positions(T, s, alpha, sink))
        assert rkv.storage_bytes(cfg)[0] == R * 2048, (T, s, alpha, sink)
        # an explicit capacity at least that large is kept as given
        big = rkv.Config(**{**cfg.__dict__, "max_refs": R + 7})
        assert rkv.storage_bytes(big)[0] == (R + 7) * 2048


def test_library_schedule_equals_the_oracle_schedule(built):
    """The positions the library tells callers to append as references are the
    oracle's schedule (ResidualKV notes §2.6), fixed and dynamic."""
    import residual_kv_cache_gb300 as rkv
    from oracle import codec as C
    for T, s, alpha, sink in ((256, 8, 0.0, 0), (32768, 16, 0.0, 0), (1000, 10, 0.1, 4),
                              (261885, 10, 0.02, 0), (261885, 10, 0.001, 0), (4096, 16, 0.02, 4),
                              (50, 7, 0.0, 60), (10000, 3, 0.7, 1)):
        cfg = rkv.Config(n_kv_heads=8, head_dim=128, d_c=512, d_ff=1536, ref_stride=s,
                         max_tokens=T, ref_alpha=alpha, ref_sink=sink)
        got = rkv.reference_positions(cfg)
        assert got.tolist() == C.reference_positions(T, s, alpha, sink).tolist(), (T, s, alpha, sink)
    L = rkv.lib()
    n = rkv._I32(0)
    assert L.rkv_reference_positions(None, None, 0, rkv.ctypes.byref(n)) == -1
    assert L.rkv_reference_positions(rkv.ctypes.byref(cfg.to_c()), None, 5, rkv.ctypes.byref(n)) == -1


def test_null_context_is_rejected(built):
    import residual_kv_cache_gb300 as rkv
    L = rkv.lib()
    assert L.rkv_reconstruct(None, None, None, 0, None, None, None) == -1
    assert b"ctx" in L.rkv_last_error()
    L.rkv_free(None)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import residual_kv_cache_gb300 as rkv
    monkeypatch.setattr(rkv, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(rkv, "_lib", None)
    with pytest.raises(rkv.RkvLibraryMissing):
        rkv.lib()


def test_output_buffers_are_checked_before_any_call():
    """A caller's output tensor must be CUDA, contiguous, of the output dtype and large
    enough; anything else is refused on the host (no device write past its end)."""
    import torch
    from residual_kv_cache_gb300 import _check_out
    with pytest.raises(ValueError):
        _check_out(torch.empty(10, dtype=torch.bfloat16), 10, torch.bfloat16, "k_out")  # CPU
    with pytest.raises(ValueError):
        _check_out(None, 10, torch.bfloat16, "k_out")
    with pytest.raises(ValueError):
        _check_out(torch.empty(10, dtype=torch.float32), 10, torch.bfloat16, "k_out")


def test_write_rows_are_checked_before_any_call():
    """The rows a write reads: the configured dtype, unit element stride, and every index
    below the tensor's row count (the library cannot see that count)."""
    import numpy as np
    import torch
    from residual_kv_cache_gb300 import _check_kv_rows
    kv = torch.zeros(256, 256, dtype=torch.float32)
    ok = dict(need_cuda=False)
    _check_kv_rows(kv, 256, torch.float32, 1, None, **ok)                    # rows 0 .. n-1
    _check_kv_rows(kv, 256, torch.float32, 3, np.array([0, 17, 255], np.int32), **ok)
    _check_kv_rows(kv.view(-1)[1:1 + 255 * 256].view(255, 256), 256, torch.float32, 1, None, **ok)
    _check_kv_rows(kv, 256, torch.float32, 1, np.array([-1], np.int32), **ok)  # the library's
    with pytest.raises(ValueError):
        _check_kv_rows(kv.to(torch.bfloat16), 256, torch.float32, 1, None, **ok)
    with pytest.raises(ValueError):
        _check_kv_rows(kv, 256, torch.float32, 2, np.array([0, 256], np.int32), **ok)
    with pytest.raises(ValueError):
        _check_kv_rows(kv, 256, torch.float32, 300, None, **ok)
    with pytest.raises(ValueError):
        _check_kv_rows(kv.t(), 256, torch.float32, 1, None, **ok)
    with pytest.raises(ValueError):
        _check_kv_rows(kv, 256, torch.float32, 1, None)                      # not on the GPU


def test_retrieve_noalloc_binding_rejects_bad_arguments():
    """The binding checks what the library cannot see (dtypes, contiguity, lengths)
    before any call: CPU tensors, a strided query view, an fp32 pool and short position
    arrays are refused with ValueError."""
    import torch
    import residual_kv_cache_gb300 as rkv
    n, d, R = 4, 64, 8
    q = torch.zeros((n, d), dtype=torch.bfloat16)
    args = dict(q_pos=torch.zeros(n, dtype=torch.int32), pool=torch.zeros((R, d), dtype=torch.bfloat16),
                pool_norm2=torch.zeros(R), pool_pos=torch.zeros(R, dtype=torch.int32))
    with pytest.raises(ValueError):
        rkv.retrieve_noalloc(q, **args)                                  # not CUDA tensors
    with pytest.raises(ValueError):
        rkv.retrieve_noalloc(torch.zeros((n, 2 * d), dtype=torch.bfloat16)[:, :d], **args)
    with pytest.raises(ValueError):
        rkv.retrieve_noalloc(q, **{**args, "pool": torch.zeros((R, d))})
    with pytest.raises(ValueError):
        rkv.retrieve_noalloc(q, **{**args, "q_pos": torch.zeros(n - 1, dtype=torch.int32)})
