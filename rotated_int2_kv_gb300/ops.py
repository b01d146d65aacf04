"""ctypes binding of liboscar.so (include/oscar.h): argument marshalling only.

Every step of the append and decode paths runs in the library's CUDA kernels;
this module only checks tensor shapes / dtypes / devices, passes raw pointers
and the current CUDA stream, and turns error codes into exceptions.  There is
no fallback: if liboscar.so is missing the import of the library fails loudly.
"""

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboscar.so")

OSCAR_OK = 0
ERR_NAMES = {-1: "OSCAR_ERR_ARG", -2: "OSCAR_ERR_NULL", -3: "OSCAR_ERR_WORKSPACE",
             -4: "OSCAR_ERR_CUDA", -5: "OSCAR_ERR_NUMERIC"}
DTYPE_BF16 = 0
DTYPE_F32 = 1
SCALE_F16 = 0     # (s, z) stored as fp16 pairs
SCALE_E4M3 = 1    # (s, z) stored as float8 E4M3 pairs
DEV_BAD_SLOT, DEV_BAD_LEN, DEV_BAD_REQ, DEV_TIMEOUT = 1, 2, 4, 8


class OscarError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s (%d): %s" % (ERR_NAMES.get(code, "?"), code, msg))
        self.code = code


class CConfig(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("sink", ctypes.c_int32), ("recent", ctypes.c_int32),
                ("clip_ratio", ctypes.c_float), ("kv_dtype", ctypes.c_int32),
                ("q_dtype", ctypes.c_int32), ("scale_dtype", ctypes.c_int32)]


class CLayerCache(ctypes.Structure):
    _fields_ = [("records", ctypes.c_void_p), ("sink", ctypes.c_void_p),
                ("recent", ctypes.c_void_p), ("rot_k", ctypes.c_void_p),
                ("rot_v", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("max_reqs", ctypes.c_int32)]


_lib = None

_SIGS = {
    "oscar_version": ([], ctypes.c_char_p),
    "oscar_last_error": ([], ctypes.c_char_p),
    "oscar_record_bytes": ([ctypes.POINTER(CConfig), ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "oscar_slot_bytes": ([ctypes.POINTER(CConfig), ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "oscar_cache_bytes_per_token": ([ctypes.POINTER(CConfig), ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "oscar_covariance": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "oscar_value_covariance": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "oscar_build_rotation": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "oscar_quantize_append": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                               ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_workspace_bytes": ([ctypes.POINTER(CConfig), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "oscar_decode_attention": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_step": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                           ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_attention_simt": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_decode_attention_noalloc": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p],
                                       ctypes.c_int),
    "oscar_covariance_workspace_bytes": ([ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
                                         ctypes.c_int),
    "oscar_covariance_device": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_value_covariance_workspace_bytes": ([ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                               ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "oscar_value_covariance_device": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_build_rotation_ex": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "oscar_prefill_workspace_bytes": ([ctypes.POINTER(CConfig), ctypes.c_int32, ctypes.c_int64,
                                       ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "oscar_prefill_attention": ([ctypes.POINTER(CConfig), ctypes.POINTER(CLayerCache), ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "oscar_device_status": ([ctypes.POINTER(ctypes.c_int32), ctypes.c_int32], ctypes.c_int),
    "oscar_selftest_bounded_wait": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "oscar_profile_enable": ([ctypes.c_int32], ctypes.c_int),
    "oscar_profile_read": ([ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                            ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
}


def lib():
    """The loaded liboscar.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("liboscar.so is not built (run __graft_entry__.build() or "
                               "python rotated_int2_kv_gb300/build.py)")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(rc):
    if rc != OSCAR_OK:
        raise OscarError(rc, lib().oscar_last_error().decode())


def last_error():
    return lib().oscar_last_error().decode()


@dataclass
class Config:
    head_dim: int
    num_q_heads: int
    num_kv_heads: int
    group_size: int = 64
    sink: int = 64
    recent: int = 256
    clip_ratio: float = 0.9
    kv_dtype: torch.dtype = torch.bfloat16
    q_dtype: torch.dtype = torch.bfloat16
    scale_fmt: str = "f16"          # "f16" or "e4m3": storage of each group's (s, z)

    def c(self):
        # the C struct is rebuilt only when a field changed since the last call
        key = (self.head_dim, self.num_q_heads, self.num_kv_heads, self.group_size, self.sink, self.recent,
               self.clip_ratio, self.kv_dtype, self.q_dtype, self.scale_fmt)
        memo = self.__dict__.get("_c_memo")
        if memo is not None and memo[0] == key:
            return memo[1]

        def code(dt):
            if dt == torch.bfloat16:
                return DTYPE_BF16
            if dt == torch.float32:
                return DTYPE_F32
            raise ValueError("dtype must be torch.bfloat16 or torch.float32")
        if self.scale_fmt not in ("f16", "e4m3"):
            raise ValueError("scale_fmt must be 'f16' or 'e4m3'")
        cc = CConfig(self.head_dim, self.num_q_heads, self.num_kv_heads, self.group_size,
                     self.sink, self.recent, self.clip_ratio, code(self.kv_dtype),
                     code(self.q_dtype), SCALE_E4M3 if self.scale_fmt == "e4m3" else SCALE_F16)
        self.__dict__["_c_memo"] = (key, cc)
        return cc

    @property
    def gqa(self):
        return self.num_q_heads // self.num_kv_heads


def version():
    return lib().oscar_version().decode()


def record_bytes(cfg):
    out = ctypes.c_int64()
    _check(lib().oscar_record_bytes(ctypes.byref(cfg.c()), ctypes.byref(out)))
    return out.value


def slot_bytes(cfg):
    out = ctypes.c_int64()
    _check(lib().oscar_slot_bytes(ctypes.byref(cfg.c()), ctypes.byref(out)))
    return out.value


def cache_bytes_per_token(cfg):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().oscar_cache_bytes_per_token(ctypes.byref(cfg.c()), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


# -- host rotation construction ---------------------------------------------

def covariance(samples):
    X = np.ascontiguousarray(samples, dtype=np.float64)
    n, d = X.shape
    C = np.empty((d, d), np.float64)
    _check(lib().oscar_covariance(X.ctypes.data, n, d, C.ctypes.data))
    return C


def value_covariance(scores, values):
    S = np.ascontiguousarray(scores, dtype=np.float64)
    V = np.ascontiguousarray(values, dtype=np.float64)
    C = np.empty((V.shape[1], V.shape[1]), np.float64)
    _check(lib().oscar_value_covariance(S.ctypes.data, V.ctypes.data, S.shape[0], S.shape[1],
                                        V.shape[1], C.ctypes.data))
    return C


def build_rotation(cov, d, use_bitrev=True, hadamard_block=None):
    """Returns (R fp32, R fp64, eigenvalues) as NumPy arrays (host).
    hadamard_block: block size of a block-diagonal Hadamard factor (None: d)."""
    R32 = np.empty((d, d), np.float32)
    R64 = np.empty((d, d), np.float64)
    w = np.empty(d, np.float64)
    cp = None
    if cov is not None:
        cov = np.ascontiguousarray(cov, dtype=np.float64)
        cp = cov.ctypes.data
    blk = d if hadamard_block is None else int(hadamard_block)
    _check(lib().oscar_build_rotation_ex(cp, d, int(bool(use_bitrev)), blk, R32.ctypes.data,
                                         R64.ctypes.data, w.ctypes.data))
    return R32, R64, w


def _act_dtype(t, name):
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise ValueError("%s must be bfloat16 or float32" % name)


def covariance_device(x, stream=None):
    """C = XᵀX / n of the rows of x (n, d) on its CUDA device: (d, d) float64."""
    if x.dim() != 2:
        raise ValueError("x must be (n, d)")
    n, d = x.shape
    dt = _act_dtype(x, "x")
    with torch.cuda.device(x.device):
        nb = ctypes.c_size_t()
        _check(lib().oscar_covariance_workspace_bytes(n, d, ctypes.byref(nb)))
        ws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=x.device)
        cov = torch.empty((d, d), dtype=torch.float64, device=x.device)
        _check(lib().oscar_covariance_device(_ptr(x, None, "x"), dt, n, d, cov.data_ptr(), ws.data_ptr(),
                                             ws.numel(), _stream(stream, x.device)))
    return cov


def value_covariance_device(scores, values, stream=None):
    """C_S = (S V)ᵀ(S V) / n_q for scores (n_q, n_k) float32 and values (n_k, d): (d, d) float64."""
    if scores.dim() != 2 or values.dim() != 2 or scores.shape[1] != values.shape[0]:
        raise ValueError("scores (n_q, n_k) and values (n_k, d) required")
    if values.device != scores.device:
        raise ValueError("scores and values must be on one device")
    n_q, n_k = scores.shape
    d = values.shape[1]
    dt = _act_dtype(values, "values")
    with torch.cuda.device(scores.device):
        nb = ctypes.c_size_t()
        _check(lib().oscar_value_covariance_workspace_bytes(n_q, n_k, d, ctypes.byref(nb)))
        ws = torch.empty(max(nb.value, 256), dtype=torch.uint8, device=scores.device)
        cov = torch.empty((d, d), dtype=torch.float64, device=scores.device)
        _check(lib().oscar_value_covariance_device(_ptr(scores, torch.float32, "scores"), _ptr(values, None, "values"),
                                                   dt, n_q, n_k, d, cov.data_ptr(), ws.data_ptr(), ws.numel(),
                                                   _stream(stream, scores.device)))
    return cov


# -- device cache -------------------------------------------------------------

class LayerCache:
    """Device buffers of one layer (allocated with PyTorch, owned here).

    records: (num_slots, Hkv, rec_bytes) uint8 with fp16 (s, z), where a slot
    is exactly the records of its KV heads; (num_slots, slot_bytes) with E4M3
    (s, z), whose slots carry padding after the packed records (head_records()
    gives the per-head view of either)."""

    def __init__(self, cfg, num_slots, max_reqs, rot_k, rot_v, device="cuda"):
        self.cfg = cfg
        rb = record_bytes(cfg)
        sb = slot_bytes(cfg)
        H, d = cfg.num_kv_heads, cfg.head_dim
        shape = (num_slots, H, rb) if sb == H * rb else (num_slots, sb)
        self.records = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.rec_bytes = rb
        self.slot_bytes = sb
        self.sink = torch.zeros((max_reqs, max(cfg.sink, 1), H, 2, d), dtype=torch.bfloat16, device=device)
        self.recent = torch.zeros((max_reqs, cfg.recent, H, 2, d), dtype=torch.bfloat16, device=device)
        self.rot_k = torch.as_tensor(np.ascontiguousarray(rot_k, np.float32)).to(device)
        self.rot_v = torch.as_tensor(np.ascontiguousarray(rot_v, np.float32)).to(device)
        self.num_slots = num_slots
        self.max_reqs = max_reqs

    def head_records(self):
        """(num_slots, Hkv, rec_bytes) view of the records."""
        H, rb = self.cfg.num_kv_heads, self.rec_bytes
        if self.records.dim() == 3:
            return self.records
        return self.records.as_strided((self.num_slots, H, rb), (self.slot_bytes, rb, 1))

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_c_struct":                      # any new buffer or size: rebuild the C struct
            object.__setattr__(self, "_c_struct", None)

    def c(self):
        cs = self.__dict__.get("_c_struct")
        if cs is None:
            cs = CLayerCache(self.records.data_ptr(), self.sink.data_ptr(), self.recent.data_ptr(),
                             self.rot_k.data_ptr(), self.rot_v.data_ptr(), self.num_slots, self.max_reqs)
            object.__setattr__(self, "_c_struct", cs)
        return cs


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None):
    if stream is None and _raw_stream is not None:   # the current stream's handle, no Stream object
        idx = device.index if device is not None and device.index is not None else torch.cuda.current_device()
        return ctypes.c_void_p(_raw_stream(idx))
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _device_of(cache, *tensors):
    """The one CUDA device that holds the cache and every given tensor; the
    library launches on the current device, so the calls below make it current."""
    di = cache.records.get_device()                  # device index (-1 for a CPU tensor)
    for t in tensors:
        if t is not None and t.get_device() != di:
            raise ValueError("all tensors must be on the cache's device %s (got %s)" % (cache.records.device, t.device))
    return cache.records.device


def quantize_append(cache, k, v, cu_new, start_pos, page_table, req_idx=None, stream=None):
    """Appends new rows k, v: (T, Hkv, d) for a batch; see oscar_quantize_append."""
    cfg = cache.cfg
    T = k.shape[0]
    if k.shape != v.shape or k.dim() != 3:
        raise ValueError("k and v must both be (T, Hkv, d)")
    B = start_pos.shape[0]
    if cu_new.shape[0] != B + 1:
        raise ValueError("cu_new must have batch + 1 entries")
    dev = _device_of(cache, k, v, cu_new, start_pos, page_table, req_idx)
    with torch.cuda.device(dev):
        _check(lib().oscar_quantize_append(
            ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(k, cfg.kv_dtype, "k"),
            _ptr(v, cfg.kv_dtype, "v"), T, _ptr(cu_new, torch.int32, "cu_new"),
            _ptr(start_pos, torch.int32, "start_pos"), _ptr(req_idx, torch.int32, "req_idx"),
            _ptr(page_table, torch.int32, "page_table"), page_table.shape[1], B, _stream(stream, dev)))


def decode_workspace_bytes(cfg, batch, max_seq_len):
    out = ctypes.c_size_t()
    _check(lib().oscar_decode_workspace_bytes(ctypes.byref(cfg.c()), batch, max_seq_len, ctypes.byref(out)))
    return out.value


def alloc_workspace(cfg, batch, max_seq_len, device="cuda"):
    n = decode_workspace_bytes(cfg, batch, max_seq_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def decode_attention(cache, q, page_table, seq_lens, max_seq_len, workspace, req_idx=None, out=None,
                     stream=None, impl="auto"):
    """One decode step: q (B, Hq, d) -> out (B, Hq, d) fp32.  impl: 'auto' or 'simt'."""
    cfg = cache.cfg
    B = q.shape[0]
    if out is None:
        out = torch.empty((B, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=q.device)
    fn = lib().oscar_decode_attention if impl == "auto" else lib().oscar_decode_attention_simt
    dev = _device_of(cache, q, page_table, seq_lens, req_idx, out, workspace)
    with torch.cuda.device(dev):
        _check(fn(ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(q, cfg.q_dtype, "q"),
                  _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                  _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(req_idx, torch.int32, "req_idx"), B,
                  max_seq_len, _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
                  workspace.numel(), _stream(stream, dev)))
    return out


def decode_step(cache, k_new, v_new, q, page_table, seq_lens, max_seq_len, workspace, req_idx=None, out=None,
                stream=None):
    """Fused decode step (oscar_decode_step): append k_new, v_new (B, Hkv, d), request b's
    token at position seq_lens[b] - 1, then attend with q (B, Hq, d) -> out (B, Hq, d) fp32."""
    cfg = cache.cfg
    B = q.shape[0]
    if k_new.shape[0] != B or v_new.shape[0] != B:
        raise ValueError("k_new and v_new need one row per request")
    dev = _device_of(cache, k_new, v_new, q, page_table, seq_lens, req_idx, out, workspace)
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty((B, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
        _check(lib().oscar_decode_step(
            ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(k_new, cfg.kv_dtype, "k_new"),
            _ptr(v_new, cfg.kv_dtype, "v_new"), _ptr(q, cfg.q_dtype, "q"), _ptr(page_table, torch.int32, "page_table"),
            page_table.shape[1], _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(req_idx, torch.int32, "req_idx"), B,
            max_seq_len, _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
            workspace.numel(), _stream(stream, dev)))
    return out


def prefill_workspace_bytes(cfg, batch, total_q):
    out = ctypes.c_size_t()
    _check(lib().oscar_prefill_workspace_bytes(ctypes.byref(cfg.c()), batch, total_q, ctypes.byref(out)))
    return out.value


def prefill_attention(cache, q, k, v, cu_q, start_pos, page_table, max_chunk, req_idx=None, out=None,
                      workspace=None, stream=None):
    """Attention of prefill chunks over the cached prefix (see oscar_prefill_attention):
    q (T, Hq, d), k, v (T, Hkv, d) -> out (T, Hq, d) fp32."""
    cfg = cache.cfg
    T = q.shape[0]
    B = start_pos.shape[0]
    if cu_q.shape[0] != B + 1:
        raise ValueError("cu_q must have batch + 1 entries")
    dev = _device_of(cache, q, k, v, cu_q, start_pos, page_table, req_idx, out, workspace)
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty((T, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty(max(prefill_workspace_bytes(cfg, B, T), 256), dtype=torch.uint8, device=dev)
        _check(lib().oscar_prefill_attention(
            ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(q, cfg.q_dtype, "q"), _ptr(k, cfg.kv_dtype, "k"),
            _ptr(v, cfg.kv_dtype, "v"), T, _ptr(cu_q, torch.int32, "cu_q"), _ptr(start_pos, torch.int32, "start_pos"),
            _ptr(req_idx, torch.int32, "req_idx"), _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
            B, int(max_chunk), _ptr(out, torch.float32, "out"), _ptr(workspace, torch.uint8, "workspace"),
            workspace.numel(), _stream(stream, dev)))
    return out


def device_status(clear=True):
    f = ctypes.c_int32()
    _check(lib().oscar_device_status(ctypes.byref(f), int(bool(clear))))
    return f.value


def selftest_bounded_wait(budget_cycles, complete, stream=None):
    """Runs the bounded mbarrier wait once (see oscar_selftest_bounded_wait)."""
    _check(lib().oscar_selftest_bounded_wait(int(budget_cycles), int(bool(complete)), _stream(stream)))


PROF_HISTORY, PROF_QUANTIZE, PROF_WINDOW_COPY, PROF_PREP, PROF_WINDOW, PROF_COMBINE, PROF_PREFILL = 0, 1, 2, 3, 4, 5, 6
PROF_STEP_PRE = 7


def profile_enable(kinds=(PROF_HISTORY,)):
    """Start event timing of the given kernel kinds (None or () stops it); clears old records."""
    mask = 0
    for k in kinds or ():
        mask |= 1 << int(k)
    _check(lib().oscar_profile_enable(mask))


def profile_read(kind):
    """(total milliseconds, launches) of kernel `kind` (0: decode history, 1: append quantise)."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(lib().oscar_profile_read(kind, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def decode_attention_noalloc(cache, q, page_table, seq_lens, max_seq_len, req_idx=None, out=None, stream=None):
    """Decode step with the library's built-in scratch (no workspace, nothing
    allocated by the library), on the device that holds q and the cache."""
    cfg = cache.cfg
    B = q.shape[0]
    if out is None:
        out = torch.empty((B, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=q.device)
    dev = _device_of(cache, q, page_table, seq_lens, req_idx, out)
    with torch.cuda.device(dev):
        _check(lib().oscar_decode_attention_noalloc(
            ctypes.byref(cfg.c()), ctypes.byref(cache.c()), _ptr(q, cfg.q_dtype, "q"),
            _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
            _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(req_idx, torch.int32, "req_idx"), B, max_seq_len,
            _ptr(out, torch.float32, "out"), _stream(stream, dev)))
    return out
