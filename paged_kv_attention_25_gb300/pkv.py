"""Thin Python binding of the pkv C ABI (include/pkv.h).

Argument marshalling only: tensors are checked (device, dtype, contiguity)
and their data pointers, the current CUDA stream and host copies of the
metadata are handed to the C library, whose kernels do all of the work.
PyTorch supplies device memory (pool storage, outputs, workspace) and streams.

The functions carry the C names (pkv_pool_create, pkv_append,
pkv_paged_attn, pkv_swap_out, pkv_swap_in, ...).  If the compiled library is
missing, every call raises RuntimeError: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
PKV_EINVAL = 1
PKV_ENOMEM = 2
PKV_ECUDA = 3
PKV_ETIMEOUT = 4
PKV_EDEVICE = 5
PKV_EUNSUPPORTED = 6
PKV_DEVERR_BLOCK_ID = 1
PKV_DEVERR_POSITION = 2
PKV_DEVERR_TIMEOUT = 4
PKV_DEVERR_INTERNAL = 8
PKV_DEBUG_WAIT_LIMIT_NS = 1
PKV_DEBUG_WITHHOLD_COPY = 2
PKV_DEBUG_FUSED_FORM = 3

KERNELS = ("append", "split_kv", "tensor_core", "merge", "swap")

# Every symbol include/pkv.h declares (checked by the CPU test suite).
EXPORTED = (
    "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_kv_ptrs", "pkv_append",
    "pkv_paged_attn_workspace_size", "pkv_paged_attn", "pkv_append_paged_attn", "pkv_paged_attn_static",
    "pkv_last_plan_stats",
    "pkv_plan_inspect", "pkv_swap_out", "pkv_swap_in", "pkv_swap_in_ahead", "pkv_swap_in_finish",
    "pkv_check_device_errors",
    "pkv_profile_enable", "pkv_profile_read", "pkv_device_sm_count", "pkv_last_error",
    "pkv_version", "pkv_copy_to_device", "pkv_copy_to_host", "pkv_debug_set",
    "pkv_cache_create", "pkv_cache_destroy", "pkv_cache_step", "pkv_cache_release", "pkv_cache_free_blocks",
)


class PkvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"pkv error {code}: {msg}")
        self.code = code


PKV_DTYPE_BF16 = 0
PKV_DTYPE_FP8_E4M3 = 1


class pkv_pool_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("k_storage", ctypes.c_void_p),
                ("v_storage", ctypes.c_void_p), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class pkv_host_meta(ctypes.Structure):
    _fields_ = [("cu_q_lens", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p), ("q_positions", ctypes.c_void_p)]


class pkv_plan_stats(ctypes.Structure):
    _fields_ = [("num_decode_items", ctypes.c_int), ("num_tc_items", ctypes.c_int),
                ("num_merge_items", ctypes.c_int), ("num_partial_rows", ctypes.c_int),
                ("decode_kv_bytes", ctypes.c_int64), ("tc_kv_bytes", ctypes.c_int64),
                ("decode_flops", ctypes.c_int64), ("tc_flops", ctypes.c_int64),
                ("decode_io_bytes", ctypes.c_int64), ("tc_io_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("plans_built", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class pkv_profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int * 5), ("total_ms", ctypes.c_double * 5)]


class pkv_work_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "req", "kv_head", "q_start", "q_count", "kv_start", "kv_end", "part", "q_count2",
                 "pos_max0", "pos_min0", "pos_max1", "pos_min1")]


_lib = None
_lock = threading.Lock()


def load_library():
    """Load libpkv.so (built by paged_kv_attention_25_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run `python -c \"import __graft_entry__ as g; g.build()\"`)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        sig = {
            "pkv_pool_create": [ctypes.POINTER(pkv_pool_desc), ctypes.POINTER(P)],
            "pkv_pool_destroy": [P],
            "pkv_pool_kv_ptrs": [P, ctypes.POINTER(P), ctypes.POINTER(P)],
            "pkv_append": [P, P, I, I, P, P, P, P, I, P],
            "pkv_paged_attn_workspace_size": [P, I, I, I, ctypes.POINTER(pkv_host_meta),
                                              ctypes.POINTER(ctypes.c_size_t)],
            "pkv_paged_attn": [P, P, I, P, P, I, P, P, I, I, ctypes.POINTER(pkv_host_meta), F, P, P, P,
                               ctypes.c_size_t, P],
            "pkv_append_paged_attn": [P, P, I, P, P, I, P, P, I, I, ctypes.POINTER(pkv_host_meta), P, P, F, P, P, P,
                                      ctypes.c_size_t, P],
            "pkv_paged_attn_static": [P, P, I, P, P, I, P, P, I, I, ctypes.POINTER(pkv_host_meta), F, P, P, P],
            "pkv_last_plan_stats": [P, ctypes.POINTER(pkv_plan_stats)],
            "pkv_plan_inspect": [I, I, I, I, I, I, ctypes.POINTER(pkv_host_meta), ctypes.POINTER(pkv_work_desc),
                                 I, ctypes.POINTER(I), ctypes.POINTER(pkv_plan_stats)],
            "pkv_swap_out": [P, P, I, P, P],
            "pkv_swap_in": [P, P, I, P, P],
            "pkv_swap_in_ahead": [P, P, I, P, P, P],
            "pkv_swap_in_finish": [P, P],
            "pkv_check_device_errors": [P, P, ctypes.POINTER(ctypes.c_uint)],
            "pkv_profile_enable": [P, I],
            "pkv_debug_set": [P, I, ctypes.c_int64],
            "pkv_profile_read": [P, ctypes.POINTER(pkv_profile), I],
            "pkv_device_sm_count": [ctypes.POINTER(I)],
            "pkv_copy_to_device": [P, P, ctypes.c_size_t, P],
            "pkv_copy_to_host": [P, P, ctypes.c_size_t, P],
            "pkv_cache_create": [I, I, F, ctypes.POINTER(P)],
            "pkv_cache_destroy": [P],
            "pkv_cache_step": [P, P, P, I, P, I, P, P, P, ctypes.POINTER(I), P, ctypes.POINTER(I), I],
            "pkv_cache_release": [P, I],
            "pkv_cache_free_blocks": [P, ctypes.POINTER(I), ctypes.POINTER(I)],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_version.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        _lib = lib
        return lib


def pkv_last_error() -> str:
    return load_library().pkv_last_error().decode()


def _check(rc: int):
    if rc != PKV_OK:
        raise PkvError(rc, pkv_last_error())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev_i32(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def _dev_bf16(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    return t


def _host_i32(a):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


class HostMeta:
    """Host copies of cu_q_lens, ctx_lens and (optionally) q_positions for planning."""

    def __init__(self, cu_q_lens, ctx_lens, q_positions=None):
        self.cu_q_lens = _host_i32(cu_q_lens)
        self.ctx_lens = _host_i32(ctx_lens)
        self.q_positions = _host_i32(q_positions)
        self.c = pkv_host_meta(self.cu_q_lens.ctypes.data, self.ctx_lens.ctypes.data,
                               None if self.q_positions is None else self.q_positions.ctypes.data)


class Pool:
    """A KV block pool: K and V storage [num_blocks, num_kv_heads, 16, head_dim] in torch memory, bf16
    (dtype "bf16") or E4M3 codes as uint8 (dtype "fp8_e4m3", values code * k_scale / code * v_scale)."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, block_size: int = 16,
                 device=None, k_storage: torch.Tensor | None = None, v_storage: torch.Tensor | None = None,
                 dtype: str = "bf16", k_scale: float = 1.0, v_scale: float = 1.0):
        lib = load_library()
        if dtype not in ("bf16", "fp8_e4m3"):
            raise ValueError("dtype must be 'bf16' or 'fp8_e4m3'")
        fp8 = dtype == "fp8_e4m3"
        tdtype = torch.uint8 if fp8 else torch.bfloat16
        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        if k_storage is None:
            k_storage = torch.zeros(shape, dtype=tdtype, device=device)
            v_storage = torch.zeros(shape, dtype=tdtype, device=device)
        for t, n in ((k_storage, "k_storage"), (v_storage, "v_storage")):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == tdtype and t.is_contiguous()):
                raise TypeError(f"{n} must be a contiguous {tdtype} CUDA tensor")
            if tuple(t.shape) != shape:
                raise ValueError(f"{n} must have shape {shape}")
        self.k, self.v = k_storage, v_storage
        self.num_blocks, self.num_kv_heads, self.head_dim, self.block_size = num_blocks, num_kv_heads, head_dim, block_size
        self.dtype, self.elem_bytes = dtype, (1 if fp8 else 2)
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        desc = pkv_pool_desc(num_blocks, block_size, num_kv_heads, head_dim,
                             PKV_DTYPE_FP8_E4M3 if fp8 else PKV_DTYPE_BF16, self.k.data_ptr(), self.v.data_ptr(),
                             self.k_scale, self.v_scale)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.k.device):
            _check(lib.pkv_pool_create(ctypes.byref(desc), ctypes.byref(h)))
        self.handle = h
        self._ws = None

    def close(self):
        if getattr(self, "handle", None):
            load_library().pkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, nbytes: int) -> torch.Tensor:
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.k.device)
        return self._ws


def pkv_pool_create(num_blocks, num_kv_heads, head_dim, block_size=16, **kw) -> Pool:
    return Pool(num_blocks, num_kv_heads, head_dim, block_size, **kw)


def pkv_pool_destroy(pool: Pool):
    pool.close()


def pkv_append(pool: Pool, block_tables, cu_q_lens, positions, k_new, v_new, stream=None):
    """Scatter k_new / v_new [T, Hkv, D] into the pool at each token's block-table slot."""
    _dev_i32(block_tables, "block_tables")
    _dev_i32(cu_q_lens, "cu_q_lens")
    _dev_i32(positions, "positions")
    _dev_bf16(k_new, "k_new")
    _dev_bf16(v_new, "v_new")
    T = positions.shape[0]
    if k_new.shape != (T, pool.num_kv_heads, pool.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [T, num_kv_heads, head_dim]")
    _check(load_library().pkv_append(pool.handle, _ptr(block_tables), block_tables.shape[1],
                                      cu_q_lens.shape[0] - 1, _ptr(cu_q_lens), _ptr(positions), _ptr(k_new),
                                      _ptr(v_new), T, _stream(stream)))


def pkv_paged_attn_workspace_size(pool: Pool, num_q_heads: int, meta: HostMeta) -> int:
    n = ctypes.c_size_t()
    R = meta.ctx_lens.shape[0]
    T = int(meta.cu_q_lens[-1])
    _check(load_library().pkv_paged_attn_workspace_size(pool.handle, num_q_heads, R, T, ctypes.byref(meta.c),
                                                        ctypes.byref(n)))
    return n.value


def pkv_paged_attn(pool: Pool, q, q_positions, block_tables, ctx_lens, cu_q_lens, meta: HostMeta, scale: float,
                   out=None, lse=None, workspace=None, stream=None, want_lse=True):
    """Generalised paged attention; returns (O [T, Hq, D] bf16, LSE [T, Hq] fp32 or None)."""
    _dev_bf16(q, "q")
    _dev_i32(q_positions, "q_positions")
    _dev_i32(block_tables, "block_tables")
    _dev_i32(ctx_lens, "ctx_lens")
    _dev_i32(cu_q_lens, "cu_q_lens")
    T, Hq, D = q.shape
    R = ctx_lens.shape[0]
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    lib = load_library()
    if workspace is None:
        workspace = pool.workspace(pkv_paged_attn_workspace_size(pool, Hq, meta))
    _check(lib.pkv_paged_attn(pool.handle, _ptr(q), Hq, _ptr(q_positions), _ptr(block_tables),
                              block_tables.shape[1], _ptr(ctx_lens), _ptr(cu_q_lens), R, T, ctypes.byref(meta.c),
                              float(scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                              _stream(stream)))
    return out, lse


def pkv_append_paged_attn(pool: Pool, q, q_positions, block_tables, ctx_lens, cu_q_lens, meta: HostMeta,
                          k_new, v_new, scale: float, out=None, lse=None, workspace=None, stream=None,
                          want_lse=True):
    """pkv_append followed by pkv_paged_attn in one call (the kernels take the new K/V from k_new / v_new);
    meta must hold host q_positions.  Returns (O, LSE)."""
    _dev_bf16(q, "q")
    _dev_i32(q_positions, "q_positions")
    _dev_i32(block_tables, "block_tables")
    _dev_i32(ctx_lens, "ctx_lens")
    _dev_i32(cu_q_lens, "cu_q_lens")
    _dev_bf16(k_new, "k_new")
    _dev_bf16(v_new, "v_new")
    T, Hq, D = q.shape
    if k_new.shape != (T, pool.num_kv_heads, pool.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [T, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    lib = load_library()
    if workspace is None:
        workspace = pool.workspace(pkv_paged_attn_workspace_size(pool, Hq, meta))
    _check(lib.pkv_append_paged_attn(pool.handle, _ptr(q), Hq, _ptr(q_positions), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(ctx_lens), _ptr(cu_q_lens), ctx_lens.shape[0], T,
                                     ctypes.byref(meta.c), _ptr(k_new), _ptr(v_new), float(scale), _ptr(out),
                                     _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


PKV_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024


def pkv_paged_attn_static(pool: Pool, q, q_positions, block_tables, ctx_lens, cu_q_lens, meta: HostMeta,
                          scale: float, out=None, lse=None, stream=None, want_lse=True):
    """pkv_paged_attn without a workspace, for callers that cannot allocate device memory.

    The library keeps the work lists and split partials in a static device
    array of PKV_STATIC_SCRATCH_BYTES; larger batches raise PkvError
    (PKV_EINVAL).  Calls share that array; the library orders them on the GPU
    in call order, whatever their pools and streams.  The first call on a
    device should come before any stream capture.  (This wrapper allocates
    `out` / `lse` with torch only when they are not given.)
    """
    _dev_bf16(q, "q")
    _dev_i32(q_positions, "q_positions")
    _dev_i32(block_tables, "block_tables")
    _dev_i32(ctx_lens, "ctx_lens")
    _dev_i32(cu_q_lens, "cu_q_lens")
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    _check(load_library().pkv_paged_attn_static(pool.handle, _ptr(q), Hq, _ptr(q_positions), _ptr(block_tables),
                                                block_tables.shape[1], _ptr(ctx_lens), _ptr(cu_q_lens),
                                                ctx_lens.shape[0], T, ctypes.byref(meta.c), float(scale), _ptr(out),
                                                _ptr(lse), _stream(stream)))
    return out, lse


def pkv_last_plan_stats(pool: Pool) -> dict:
    st = pkv_plan_stats()
    _check(load_library().pkv_last_plan_stats(pool.handle, ctypes.byref(st)))
    return st.as_dict()


def pkv_plan_inspect(num_q_heads, num_kv_heads, head_dim, num_sms, meta: HostMeta, max_items=1 << 20):
    """Host-only planning: returns (structured numpy array of work items, stats dict)."""
    lib = load_library()
    R = meta.ctx_lens.shape[0]
    T = int(meta.cu_q_lens[-1])
    n = ctypes.c_int()
    st = pkv_plan_stats()
    _check(lib.pkv_plan_inspect(num_q_heads, num_kv_heads, head_dim, num_sms, R, T, ctypes.byref(meta.c), None, 0,
                                ctypes.byref(n), ctypes.byref(st)))
    items = (pkv_work_desc * max(n.value, 1))()
    _check(lib.pkv_plan_inspect(num_q_heads, num_kv_heads, head_dim, num_sms, R, T, ctypes.byref(meta.c), items,
                                n.value, ctypes.byref(n), ctypes.byref(st)))
    dt = np.dtype([(f, np.int32) for f, _ in pkv_work_desc._fields_])
    arr = np.frombuffer(bytes(items), dtype=dt, count=n.value).copy()
    return arr, st.as_dict()


def pkv_swap_out(pool: Pool, block_ids, host_buf: torch.Tensor, stream=None):
    """Copy blocks (host int32 ids) into host_buf [n, 2, Hkv, 16, D] (pinned CPU tensor)."""
    ids = _host_i32(block_ids)
    _check_host_buf(pool, host_buf, ids.shape[0])
    _check(load_library().pkv_swap_out(pool.handle, ids.ctypes.data, ids.shape[0], host_buf.data_ptr(),
                                        _stream(stream)))


class Cache:
    """Two-tier (GPU pool / CPU host slots) block manager for conversations; host only."""

    def __init__(self, gpu_blocks: int, cpu_blocks: int, token_cost: float = 0.0):
        lib = load_library()
        h = ctypes.c_void_p()
        _check(lib.pkv_cache_create(gpu_blocks, cpu_blocks, float(token_cost), ctypes.byref(h)))
        self.handle = h
        self.gpu_blocks, self.cpu_blocks = gpu_blocks, cpu_blocks

    def step(self, conv_ids, new_tokens, max_blocks: int):
        """Plan one step; returns dict(block_tables [n, max_blocks], ctx_lens, recompute,
        swap_out [k, 2] (pool block, host slot), swap_in [m, 2] (host slot, pool block))."""
        ids, nt = _host_i32(conv_ids), _host_i32(new_tokens)
        n = ids.shape[0]
        cap = self.gpu_blocks + self.cpu_blocks + 1
        bt = np.full((max(n, 1), max_blocks), -1, np.int32)
        ctx, rec = np.zeros(max(n, 1), np.int32), np.zeros(max(n, 1), np.int32)
        so, si = np.zeros((cap, 2), np.int32), np.zeros((cap, 2), np.int32)
        nso, nsi = ctypes.c_int(), ctypes.c_int()
        _check(load_library().pkv_cache_step(self.handle, ids.ctypes.data, nt.ctypes.data, n, bt.ctypes.data,
                                             max_blocks, ctx.ctypes.data, rec.ctypes.data, so.ctypes.data,
                                             ctypes.byref(nso), si.ctypes.data, ctypes.byref(nsi), cap))
        return {"block_tables": bt[:n], "ctx_lens": ctx[:n], "recompute": rec[:n],
                "swap_out": so[:nso.value].copy(), "swap_in": si[:nsi.value].copy()}

    def release(self, conv: int):
        _check(load_library().pkv_cache_release(self.handle, int(conv)))

    def free_blocks(self):
        g, c = ctypes.c_int(), ctypes.c_int()
        _check(load_library().pkv_cache_free_blocks(self.handle, ctypes.byref(g), ctypes.byref(c)))
        return g.value, c.value

    def close(self):
        if self.handle:
            load_library().pkv_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _same_bytes(a: torch.Tensor, b: torch.Tensor):
    if not (a.is_contiguous() and b.is_contiguous()):
        raise TypeError("tensors must be contiguous")
    n = a.numel() * a.element_size()
    if n != b.numel() * b.element_size():
        raise ValueError("tensors differ in size")
    return n


def pkv_copy_to_device(dst: torch.Tensor, host_src: torch.Tensor, stream=None):
    """dst (CUDA) <- host_src (CPU; pinned for an asynchronous copy), by the copy engines on `stream`."""
    if not dst.is_cuda or host_src.is_cuda:
        raise TypeError("dst must be a CUDA tensor and host_src a CPU tensor")
    _check(load_library().pkv_copy_to_device(dst.data_ptr(), host_src.data_ptr(), _same_bytes(dst, host_src),
                                             _stream(stream)))


def pkv_copy_to_host(host_dst: torch.Tensor, src: torch.Tensor, stream=None):
    """host_dst (CPU; pinned for an asynchronous copy) <- src (CUDA), by the copy engines on `stream`."""
    if host_dst.is_cuda or not src.is_cuda:
        raise TypeError("host_dst must be a CPU tensor and src a CUDA tensor")
    _check(load_library().pkv_copy_to_host(host_dst.data_ptr(), src.data_ptr(), _same_bytes(host_dst, src),
                                           _stream(stream)))


def pkv_swap_in(pool: Pool, block_ids, host_buf: torch.Tensor, stream=None):
    """Copy host_buf [n, 2, Hkv, 16, D] back into the pool blocks block_ids."""
    ids = _host_i32(block_ids)
    _check_host_buf(pool, host_buf, ids.shape[0])
    _check(load_library().pkv_swap_in(pool.handle, ids.ctypes.data, ids.shape[0], host_buf.data_ptr(),
                                       _stream(stream)))


def pkv_swap_in_ahead(pool: Pool, block_ids, host_buf: torch.Tensor, copy_stream, stream=None):
    """Start the copy-engine transfer of host_buf [n, 2, Hkv, 16, D] on copy_stream (after the work queued
    on `stream`); the blocks land in block_ids at the pool's next call or at pkv_swap_in_finish."""
    ids = _host_i32(block_ids)
    _check_host_buf(pool, host_buf, ids.shape[0])
    _check(load_library().pkv_swap_in_ahead(pool.handle, ids.ctypes.data, ids.shape[0], host_buf.data_ptr(),
                                             _stream(copy_stream), _stream(stream)))


def pkv_swap_in_finish(pool: Pool, stream=None):
    """Land a pending ahead-of-time swap-in on `stream` (no-op if none is pending)."""
    _check(load_library().pkv_swap_in_finish(pool.handle, _stream(stream)))


def _check_host_buf(pool, host_buf, n):
    if not (isinstance(host_buf, torch.Tensor) and not host_buf.is_cuda and host_buf.is_contiguous()):
        raise TypeError("host_buf must be a contiguous CPU tensor (pinned for asynchronous copies)")
    need = n * 2 * pool.num_kv_heads * pool.block_size * pool.head_dim * pool.elem_bytes
    if host_buf.numel() * host_buf.element_size() < need:
        raise ValueError(f"host_buf holds fewer than {need} bytes")


def pkv_check_device_errors(pool: Pool, stream=None) -> int:
    """Synchronise and return the device error-word bits (0 if none); clears the word."""
    flags = ctypes.c_uint()
    rc = load_library().pkv_check_device_errors(pool.handle, _stream(stream), ctypes.byref(flags))
    if rc not in (PKV_OK, PKV_EDEVICE, PKV_ETIMEOUT):
        _check(rc)
    return flags.value


def pkv_profile_enable(pool: Pool, on=True):
    """on: False/0 off, True/1 on, 2 on with the two attention kernels of a call run one after the other."""
    _check(load_library().pkv_profile_enable(pool.handle, int(on)))


def pkv_debug_set(pool: Pool, what: int, value: int):
    """Test settings: PKV_DEBUG_WAIT_LIMIT_NS (bounded-wait limit), PKV_DEBUG_WITHHOLD_COPY (0, 1, 2) or
    PKV_DEBUG_FUSED_FORM (0 per batch, 1 in-kernel append, 2 append first)."""
    _check(load_library().pkv_debug_set(pool.handle, int(what), int(value)))


def pkv_profile_read(pool: Pool, reset: bool = False) -> dict:
    p = pkv_profile()
    _check(load_library().pkv_profile_read(pool.handle, ctypes.byref(p), 1 if reset else 0))
    return {KERNELS[i]: {"launches": p.launches[i], "total_ms": p.total_ms[i]} for i in range(len(KERNELS))}


def pkv_device_sm_count() -> int:
    n = ctypes.c_int()
    _check(load_library().pkv_device_sm_count(ctypes.byref(n)))
    return n.value


def pkv_version() -> str:
    return load_library().pkv_version().decode()
