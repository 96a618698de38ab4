"""Python binding of librkv (the ResidualKV cache codec for GB300, sm_103a).

Argument marshalling only: every step of the codec runs in the CUDA library behind
the C ABI declared in ``include/rkv.h``.  PyTorch provides device memory and streams.
If ``librkv.so`` has not been built, importing works but any use raises
``RkvLibraryMissing``: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

__all__ = ["RkvError", "RkvLibraryMissing", "Config", "Codec", "lib", "LIB_PATH", "retrieve_noalloc",
           "FLAG_TIMEOUT", "FLAG_BAD_INDEX", "FLAG_UNWRITTEN", "FLAG_FP16_SAT", "FLAG_BAD_SLOT",
           "ABI_FUNCTIONS", "reconstruct_multi"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librkv.so")

RKV_F32, RKV_BF16 = 0, 1
FLAG_TIMEOUT, FLAG_BAD_INDEX, FLAG_UNWRITTEN, FLAG_FP16_SAT, FLAG_BAD_SLOT = 1, 2, 4, 8, 16
STATUS_NAMES = {0: "RKV_OK", -1: "RKV_EINVAL", -2: "RKV_EALIGN", -3: "RKV_ECAPACITY",
                -4: "RKV_EEMPTYPOOL", -5: "RKV_ECUDA", -6: "RKV_EDEVICE", -7: "RKV_ETIMEOUT"}


class RkvLibraryMissing(RuntimeError):
    pass


class RkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("d_c", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("group", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("ref_stride", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("rope_base", ctypes.c_double),
                ("batch", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("max_refs", ctypes.c_int32), ("max_rows", ctypes.c_int32),
                ("ref_alpha", ctypes.c_double), ("ref_sink", ctypes.c_int32),
                ("mean_precompute", ctypes.c_int32)]


class _Storage(ctypes.Structure):
    _fields_ = [("pool_fp8", ctypes.c_void_p), ("pool_norm2", ctypes.c_void_p),
                ("pool_pos", ctypes.c_void_p), ("codes", ctypes.c_void_p),
                ("meta", ctypes.c_void_p), ("ref_idx", ctypes.c_void_p)]


class _Timing(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


# name -> (restype, argtypes); the entry points of include/rkv.h
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
ABI_FUNCTIONS = {
    "rkv_storage_bytes": (_I32, [ctypes.POINTER(_Config), ctypes.POINTER(ctypes.c_size_t)]),
    "rkv_reference_positions": (_I32, [ctypes.POINTER(_Config), ctypes.POINTER(_I32), _I32,
                                       ctypes.POINTER(_I32)]),
    "rkv_create": (_I32, [ctypes.POINTER(_Config), _P, _P, _P, _P, ctypes.POINTER(_Storage), _P,
                          ctypes.POINTER(_P)]),
    "rkv_pool_append": (_I32, [_P, _P, _I64, _P, _P, _P, _I32, _P]),
    "rkv_compress": (_I32, [_P, _P, _I64, _P, _P, _P, _I32, _P]),
    "rkv_reconstruct": (_I32, [_P, _P, _P, _I32, _P, _P, _P]),
    "rkv_sparse_attention": (_I32, [_P, _P, _I32, _P, _P, _I32, _P, _P]),
    "rkv_restore_attend": (_I32, [_P, _P, _P, _I32, _P, _I32, _P, _P]),
    "rkv_reconstruct_multi": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _P]),
    "rkv_get_status": (_I32, [_P, ctypes.POINTER(_I32), _P]),
    "rkv_reset": (_I32, [_P, _I32, _P]),
    "rkv_pool_cache": (_I32, [_P, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "rkv_last_error": (ctypes.c_char_p, []),
    "rkv_free": (None, [_P]),
    "rkv_set_timing": (_I32, [_P, _I32]),
    "rkv_get_timing": (_I32, [_P, ctypes.POINTER(_Timing), _I32, _I32]),
    "rkv_launch_count": (_I64, [_P]),
    "rkv_debug_scratch": (_I32, [_P, _I32, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "rkv_debug_timeout_probe": (_I32, [_P, _P]),
    "rkv_retrieve_noalloc": (_I32, [_P, _P, _I32, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load librkv.so from this package's directory (built in-tree)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RkvLibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m residual_kv_cache_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in ABI_FUNCTIONS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int):
    if status != 0:
        raise RkvError(status, lib().rkv_last_error().decode(errors="replace"))


def _dtype_code(dt) -> int:
    if dt in ("fp32", torch.float32):
        return RKV_F32
    if dt in ("bf16", torch.bfloat16):
        return RKV_BF16
    raise ValueError(f"unsupported dtype {dt}")


def _host_i32(a):
    """Host int32 contiguous array (numpy) and its address; None passes NULL."""
    if a is None:
        return None, None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data


# The current stream's raw handle without building a Stream object (a few microseconds
# per call on the host, which an idle GPU waits for); the public call is the fallback.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _torch_dtype(dt):
    """torch dtype of a config dtype ("fp32" / "bf16" or the torch dtypes themselves)."""
    return torch.float32 if _dtype_code(dt) == RKV_F32 else torch.bfloat16


def _check_kv_rows(kv, d_kv: int, dtype, n: int, src, need_cuda: bool = True):
    """The rows a write call reads: a [rows, 2d_k] tensor of the configured kv dtype with
    unit element stride, and every row index it will read below `rows` (the library
    knows only the row stride, not how many rows there are).  Negative indices are left
    to the library's own check."""
    if not isinstance(kv, torch.Tensor) or kv.dim() != 2 or kv.shape[1] != d_kv \
            or (need_cuda and not kv.is_cuda):
        raise ValueError("kv must be a [rows, 2*d_k] CUDA tensor")
    if kv.dtype != dtype or kv.stride(1) != 1:
        raise ValueError(f"kv must hold {dtype} values with unit element stride")
    rows = kv.shape[0]
    if n == 0:
        return
    if src is None:
        if n > rows:
            raise ValueError("kv has fewer rows than the call writes")
    elif int(src.max()) >= rows:
        raise ValueError("src_rows must index rows of kv")


def _check_out(t, n_elems: int, dtype, what: str):
    """A caller-supplied output: a contiguous CUDA tensor of `dtype` with room for
    n_elems values (the library writes exactly that many, from its start)."""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda \
            or not t.is_contiguous() or t.numel() < n_elems:
        raise ValueError(f"{what} must be a contiguous CUDA tensor of {dtype} with at least "
                         f"{n_elems} elements")


def _stream_ptr(stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream


@dataclass
class Config:
    n_kv_heads: int
    head_dim: int
    d_c: int
    d_ff: int
    topk: int = 4
    group: int = 32
    bits: int = 4
    ref_stride: int = 16
    kv_dtype: str = "bf16"
    out_dtype: str = "bf16"
    rope_base: float = 10000.0
    batch: int = 1
    max_tokens: int = 32768
    max_refs: int = 0          # 0 -> the schedule's positions below max_tokens
    max_rows: int = 0
    ref_alpha: float = 0.0     # dynamic-stride growth; 0 = fixed stride
    ref_sink: int = 0          # sink tokens kept as references ahead of the schedule
    mean_precompute: int = 0   # 1: the mean's pre-activations from the references' own

    def to_c(self) -> _Config:
        return _Config(self.n_kv_heads, self.head_dim, self.d_c, self.d_ff, self.topk,
                       self.group, self.bits, self.ref_stride, _dtype_code(self.kv_dtype),
                       _dtype_code(self.out_dtype), float(self.rope_base), self.batch,
                       self.max_tokens, self.max_refs, self.max_rows, float(self.ref_alpha),
                       self.ref_sink, self.mean_precompute)

    @property
    def d_kv(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim


def storage_bytes(cfg: Config):
    sizes = (ctypes.c_size_t * 6)()
    c = cfg.to_c()
    _check(lib().rkv_storage_bytes(ctypes.byref(c), sizes))
    return list(sizes)


def reference_positions(cfg: Config) -> np.ndarray:
    """The schedule's reference positions below cfg.max_tokens (int32, increasing)."""
    c = cfg.to_c()
    n = _I32(0)
    _check(lib().rkv_reference_positions(ctypes.byref(c), None, 0, ctypes.byref(n)))
    out = np.empty(n.value, dtype=np.int32)
    _check(lib().rkv_reference_positions(ctypes.byref(c),
                                         out.ctypes.data_as(ctypes.POINTER(_I32)), n.value,
                                         ctypes.byref(n)))
    return out


def retrieve_noalloc(queries, q_pos, pool, pool_norm2, pool_pos, topk: int = 4, out=None,
                     flags=None, stream=None):
    """Top-k retrieval of one sequence through rkv_retrieve_noalloc (no allocation in the
    library; scratch is a fixed device array).  queries [n, d] bf16, q_pos [n] int32,
    pool [R, d] bf16, pool_norm2 [R] fp32, pool_pos [R] int32, all contiguous CUDA
    tensors (the library reads rows of exactly d elements).  Returns out [n, topk] int32
    (allocated here by torch if not given)."""
    for t, dt, what in ((queries, torch.bfloat16, "queries"), (pool, torch.bfloat16, "pool"),
                        (q_pos, torch.int32, "q_pos"), (pool_norm2, torch.float32, "pool_norm2"),
                        (pool_pos, torch.int32, "pool_pos")):
        if not isinstance(t, torch.Tensor) or t.dtype != dt or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{what} must be a contiguous CUDA tensor of {dt}")
    if queries.dim() != 2 or pool.dim() != 2 or pool.shape[1] != queries.shape[1]:
        raise ValueError("queries [n, d] and pool [R, d] must share d")
    n, d = queries.shape
    R = pool.shape[0]
    if q_pos.numel() != n:
        raise ValueError("q_pos must hold one position per query row")
    if pool_norm2.numel() < R or pool_pos.numel() < R:
        raise ValueError("pool_norm2 and pool_pos must hold one entry per pool row")
    if not 1 <= topk <= 4:
        raise ValueError("topk must be in 1..4")
    if out is None:
        out = torch.empty((n, topk), dtype=torch.int32, device=queries.device)
    _check_out(out, n * topk, torch.int32, "out")
    if flags is not None:
        _check_out(flags, 1, torch.int32, "flags")
    fp = flags.data_ptr() if flags is not None else None
    _check(lib().rkv_retrieve_noalloc(queries.data_ptr(), q_pos.data_ptr(), n, pool.data_ptr(),
                                      pool_norm2.data_ptr(), pool_pos.data_ptr(), R, d, topk,
                                      out.data_ptr(), fp, _stream_ptr(stream)))
    return out


def reconstruct_multi(codecs, seqs, poss, k_outs=None, v_outs=None, stream=None):
    """Restore each codec's selection (seqs[i], poss[i]: int32 CUDA tensors) in one launch
    (codecs of equal shape on one device).  Returns the lists (K_i, V_i)."""
    n = len(codecs)
    if n == 0 or len(seqs) != n or len(poss) != n:
        raise ValueError("one seq and pos tensor per codec")
    k_outs = list(k_outs) if k_outs is not None else [None] * n
    v_outs = list(v_outs) if v_outs is not None else [None] * n
    ns = []
    for i, (c, sq, ps) in enumerate(zip(codecs, seqs, poss)):
        for t in (sq, ps):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("seq and pos must be contiguous int32 CUDA tensors")
        m = int(ps.numel())
        if int(sq.numel()) != m:
            raise ValueError("seq and pos must have the same length")
        N, D = c.cfg.n_kv_heads, c.cfg.head_dim
        odt = _torch_dtype(c.cfg.out_dtype)
        if k_outs[i] is None:
            k_outs[i] = torch.empty((m, N, D), dtype=odt, device=c.device)
        if v_outs[i] is None:
            v_outs[i] = torch.empty((m, N, D), dtype=odt, device=c.device)
        _check_out(k_outs[i], m * N * D, odt, "k_out")
        _check_out(v_outs[i], m * N * D, odt, "v_out")
        ns.append(m)
    P = ctypes.c_void_p * n
    ctxs = P(*[c._ctx for c in codecs])
    sp, pp_ = P(*[t.data_ptr() for t in seqs]), P(*[t.data_ptr() for t in poss])
    kp, vp = P(*[t.data_ptr() for t in k_outs]), P(*[t.data_ptr() for t in v_outs])
    nsel = (_I32 * n)(*ns)
    _check(lib().rkv_reconstruct_multi(ctxs, n, sp, pp_, nsel, kp, vp, _stream_ptr(stream)))
    return k_outs, v_outs


class Codec:
    """One codec layer: caller-side storage tensors plus the library context."""

    STORAGE = ("pool_fp8", "pool_norm2", "pool_pos", "codes", "meta", "ref_idx")

    def __init__(self, cfg: Config, weights: dict, device=None, stream=None):
        self.cfg = cfg
        self.device = torch.device(device or "cuda")
        c = cfg.to_c()
        self._c = c
        sizes = (ctypes.c_size_t * 6)()
        _check(lib().rkv_storage_bytes(ctypes.byref(c), sizes))
        B, T = c.batch, c.max_tokens
        dkv, G = cfg.d_kv, cfg.d_c // cfg.group
        R = sizes[0] // (B * dkv)                      # pool slots per sequence
        cb = sizes[3] // (B * T)
        dev = self.device
        self._shape = (B, R, dkv)
        self.pool_fp8 = torch.empty((B, R, dkv), dtype=torch.uint8, device=dev)
        self.pool_norm2 = torch.empty((B, R), dtype=torch.float32, device=dev)
        self.pool_pos = torch.empty((B, R), dtype=torch.int32, device=dev)
        self.codes = torch.zeros((B, T, cb), dtype=torch.uint8, device=dev)
        self.meta = torch.zeros((B, T, G, 2), dtype=torch.float16, device=dev)
        self.ref_idx = torch.empty((B, T, cfg.topk), dtype=torch.int32, device=dev)
        st = _Storage(*(getattr(self, n).data_ptr() for n in self.STORAGE))
        w = [weights[k] for k in ("Wc1", "Wc2", "Wc3", "Wd")]
        for t in w:
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights must be contiguous bf16 CUDA tensors")
        ctx = ctypes.c_void_p()
        _check(lib().rkv_create(ctypes.byref(c), *(t.data_ptr() for t in w), ctypes.byref(st),
                                _stream_ptr(stream), ctypes.byref(ctx)))
        self._ctx = ctx

    @property
    def pool_bf16(self) -> torch.Tensor:
        """The context's bf16 copy of the pool ([B, R_cap, 2d_k], the retrieval's
        tensor-core operand; library memory, valid while the codec lives): a view, not a
        copy."""
        p, b = ctypes.c_void_p(), ctypes.c_size_t()
        _check(lib().rkv_pool_cache(self._ctx, ctypes.byref(p), ctypes.byref(b)))
        B, R, dkv = self._shape
        cai = type("_Dev", (), {})()
        cai.__cuda_array_interface__ = {"shape": (B, R, dkv), "typestr": "<u2",
                                        "data": (p.value, False), "version": 3}
        return torch.as_tensor(cai, device=self.device).view(torch.bfloat16)

    def pool_cache_bytes(self) -> int:
        p, b = ctypes.c_void_p(), ctypes.c_size_t()
        _check(lib().rkv_pool_cache(self._ctx, ctypes.byref(p), ctypes.byref(b)))
        return int(b.value)

    # -- ABI calls -------------------------------------------------------------------
    def _rows_call(self, fn, kv, seq, pos, src_rows, stream):
        seq_a, seq_p = _host_i32(seq)
        pos_a, pos_p = _host_i32(pos)
        src_a, src_p = _host_i32(src_rows)
        n = len(pos_a)
        if len(seq_a) != n or (src_a is not None and len(src_a) != n):
            raise ValueError("seq, pos and src_rows must have the same length")
        _check_kv_rows(kv, self.cfg.d_kv, _torch_dtype(self.cfg.kv_dtype), n, src_a)
        _check(fn(self._ctx, kv.data_ptr(), kv.stride(0), src_p, seq_p, pos_p, n,
                  _stream_ptr(stream)))

    def pool_append(self, kv, seq, pos, src_rows=None, stream=None):
        """Append reference rows (seq, pos: host int arrays)."""
        self._rows_call(lib().rkv_pool_append, kv, seq, pos, src_rows, stream)

    def compress(self, kv, seq, pos, src_rows=None, stream=None):
        """Encode non-reference rows (seq, pos: host int arrays)."""
        self._rows_call(lib().rkv_compress, kv, seq, pos, src_rows, stream)

    def reconstruct(self, seq, pos, k_out=None, v_out=None, stream=None):
        """Restore selected tokens; seq, pos are int32 CUDA tensors.  Returns (K, V)."""
        n = int(pos.numel())
        N, D = self.cfg.n_kv_heads, self.cfg.head_dim
        odt = _torch_dtype(self.cfg.out_dtype)
        if k_out is None:
            k_out = torch.empty((n, N, D), dtype=odt, device=self.device)
        if v_out is None:
            v_out = torch.empty((n, N, D), dtype=odt, device=self.device)
        for t in (seq, pos):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("seq and pos must be contiguous int32 CUDA tensors")
        if int(seq.numel()) != n:
            raise ValueError("seq and pos must have the same length")
        _check_out(k_out, n * N * D, odt, "k_out")
        _check_out(v_out, n * N * D, odt, "v_out")
        _check(lib().rkv_reconstruct(self._ctx, seq.data_ptr(), pos.data_ptr(), n,
                                     k_out.data_ptr(), v_out.data_ptr(), _stream_ptr(stream)))
        return k_out, v_out

    def sparse_attention(self, q, k, v, out=None, stream=None):
        """softmax(q K^T / sqrt(D)) V over the rows of k, v (a restore's outputs).
        q: [H_q, D] fp32 CUDA tensor; returns out [H_q, D] fp32."""
        N, D = self.cfg.n_kv_heads, self.cfg.head_dim
        odt = _torch_dtype(self.cfg.out_dtype)
        if q.dtype != torch.float32 or not q.is_cuda or not q.is_contiguous() or q.dim() != 2 \
                or q.shape[1] != D:
            raise ValueError("q must be a contiguous [H_q, D] fp32 CUDA tensor")
        for t in (k, v):
            if t.dtype != odt or not t.is_cuda or not t.is_contiguous() or tuple(t.shape[1:]) != (N, D):
                raise ValueError("k and v must be contiguous [n, N, D] CUDA tensors of out_dtype")
        if k.shape[0] != v.shape[0]:
            raise ValueError("k and v must have the same rows")
        if out is None:
            out = torch.empty((q.shape[0], D), dtype=torch.float32, device=q.device)
        _check_out(out, q.shape[0] * D, torch.float32, "out")
        _check(lib().rkv_sparse_attention(self._ctx, q.data_ptr(), q.shape[0], k.data_ptr(),
                                          v.data_ptr(), k.shape[0], out.data_ptr(),
                                          _stream_ptr(stream)))
        return out

    def restore_attend(self, seq, pos, q, out=None, stream=None):
        """softmax(q K_hat^T / sqrt(D)) V_hat over the selected tokens, restored on chip
        (nothing of K_hat / V_hat is written).  seq, pos: int32 CUDA tensors; q: [H_q, D]
        fp32 CUDA tensor; returns out [H_q, D] fp32."""
        D = self.cfg.head_dim
        n = int(pos.numel())
        for t in (seq, pos):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("seq and pos must be contiguous int32 CUDA tensors")
        if int(seq.numel()) != n:
            raise ValueError("seq and pos must have the same length")
        if q.dtype != torch.float32 or not q.is_cuda or not q.is_contiguous() or q.dim() != 2 \
                or q.shape[1] != D:
            raise ValueError("q must be a contiguous [H_q, D] fp32 CUDA tensor")
        if out is None:
            out = torch.empty((q.shape[0], D), dtype=torch.float32, device=q.device)
        _check_out(out, q.shape[0] * D, torch.float32, "out")
        _check(lib().rkv_restore_attend(self._ctx, seq.data_ptr(), pos.data_ptr(), n,
                                        q.data_ptr(), q.shape[0], out.data_ptr(),
                                        _stream_ptr(stream)))
        return out

    def reset(self, seq: int = -1, stream=None):
        """Empty one sequence's pool and token rows (seq = -1: all sequences)."""
        _check(lib().rkv_reset(self._ctx, seq, _stream_ptr(stream)))

    def get_status(self, stream=None) -> int:
        flags = ctypes.c_int32(0)
        st = lib().rkv_get_status(self._ctx, ctypes.byref(flags), _stream_ptr(stream))
        if st not in (0, -6, -7):
            _check(st)
        return int(flags.value)

    # -- instrumentation ---------------------------------------------------------------
    def set_timing(self, enable: bool):
        _check(lib().rkv_set_timing(self._ctx, 1 if enable else 0))

    def get_timing(self, reset: bool = False) -> dict:
        n = lib().rkv_get_timing(self._ctx, None, 0, 0)
        buf = (_Timing * max(n, 1))()
        n = lib().rkv_get_timing(self._ctx, buf, n, 1 if reset else 0)
        return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
                for i in range(n)}

    def launch_count(self) -> int:
        return int(lib().rkv_launch_count(self._ctx))

    def debug_scratch(self, which: int):
        """(device address, bytes) of a scratch tensor of the last compress pass."""
        p, b = ctypes.c_void_p(), ctypes.c_size_t()
        _check(lib().rkv_debug_scratch(self._ctx, which, ctypes.byref(p), ctypes.byref(b)))
        return p.value, b.value

    def debug_timeout_probe(self, stream=None):
        """Launch one block whose bounded wait must expire (failure-detection test)."""
        _check(lib().rkv_debug_timeout_probe(self._ctx, _stream_ptr(stream)))

    def free(self):
        if getattr(self, "_ctx", None):
            lib().rkv_free(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
