"""Thin ctypes binding of libhs.so (declared in include/hs.h).

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels.  torch is used for device memory and streams; tensors are passed
as raw pointers.  There is no CPU fallback: if the library cannot be loaded,
importing this module's ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhs.so")

HS_OK = 0
HS_ERR_INVALID = -1
HS_ERR_CONFIG = -2
HS_ERR_OOM = -3
HS_ERR_CAPACITY = -4
HS_ERR_CUDA = -5
HS_ERR_DEVICE = -6

HS_DEVERR_REQ_RANGE = 0x1
HS_DEVERR_CAPACITY = 0x2
HS_DEVERR_EMPTY = 0x4
HS_DEVERR_TIMEOUT = 0x8
HS_DEVERR_METADATA = 0x10
HS_DEVERR_NO_LEAD = 0x20

HS_K_APPEND, HS_K_SELECT, HS_K_ATTENTION, HS_K_COUNT = 0, 1, 2, 3

HS_REPLACE_LRU = 0
HS_REPLACE_FIFO = 1
HS_REPLACE_RANDOM = 2
REPLACEMENT = {"lru": HS_REPLACE_LRU, "fifo": HS_REPLACE_FIFO, "random": HS_REPLACE_RANDOM}
KERNEL_NAMES = ("append", "select", "attention")

# the symbols include/hs.h declares
EXPORTED = ("hs_create", "hs_destroy", "hs_append", "hs_decode_layer", "hs_stats", "hs_snapshot",
            "hs_reset_request", "hs_set_timing", "hs_kernel_times", "hs_last_error",
            "hs_status_string", "hs_row_elems", "hs_indexer_topk_static",
            "hs_indexer_topk_static_error")


class HsConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("max_requests", ctypes.c_int32),
                ("max_context", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
                ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32), ("shared_kv", ctypes.c_int32),
                ("d_idx", ctypes.c_int32), ("top_k", ctypes.c_int32), ("hot_slots", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("device", ctypes.c_int32),
                ("fetch_mode", ctypes.c_int32), ("replacement", ctypes.c_int32),
                ("replacement_seed", ctypes.c_uint32), ("write_allocate", ctypes.c_int32),
                ("idx_heads", ctypes.c_int32), ("index_share", ctypes.c_int32),
                ("share_prefetch", ctypes.c_int32), ("page_size", ctypes.c_int32)]


class HsStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "hits", "misses", "h2d_bytes", "d2h_bytes", "decode_calls", "append_calls",
        "host_bytes", "hot_bytes", "index_bytes", "meta_bytes", "host_huge_bytes", "full_selects",
        "att_host_wait_ns", "att_host_stages", "att_hbm_wait_ns", "att_hbm_stages", "att_last_span_ns",
        "att_last_median_ns")] + [
        ("device_error", ctypes.c_uint32), ("_pad", ctypes.c_uint32)]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_ if n != "_pad"}


class HsError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_name(status)}: {msg}")
        self.status = status


_LIB = None


def lib():
    """Load libhs.so (raises OSError when it is missing: no fallback)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with tiered_kv_cache_int8_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
        L.hs_create.argtypes = [P(HsConfig), P(VP)]
        L.hs_create.restype = ctypes.c_int
        L.hs_destroy.argtypes = [VP]
        L.hs_destroy.restype = None
        L.hs_append.argtypes = [VP, I32, I32, VP, I32, VP, VP, VP]
        L.hs_append.restype = ctypes.c_int
        L.hs_decode_layer.argtypes = [VP, I32, I32, VP, VP, VP, VP, VP, VP, VP, VP]
        L.hs_decode_layer.restype = ctypes.c_int
        L.hs_stats.argtypes = [VP, P(HsStats)]
        L.hs_stats.restype = ctypes.c_int
        L.hs_snapshot.argtypes = [VP, I32, I32, VP, I32, VP, VP, VP, VP]
        L.hs_snapshot.restype = ctypes.c_int
        L.hs_reset_request.argtypes = [VP, I32, VP]
        L.hs_reset_request.restype = ctypes.c_int
        L.hs_set_timing.argtypes = [VP, I32]
        L.hs_set_timing.restype = ctypes.c_int
        L.hs_kernel_times.argtypes = [VP, P(ctypes.c_double), P(ctypes.c_int64)]
        L.hs_kernel_times.restype = ctypes.c_int
        L.hs_last_error.argtypes = [VP]
        L.hs_last_error.restype = ctypes.c_char_p
        L.hs_status_string.argtypes = [I32]
        L.hs_status_string.restype = ctypes.c_char_p
        L.hs_row_elems.argtypes = [P(HsConfig)]
        L.hs_row_elems.restype = I32
        L.hs_indexer_topk_static.argtypes = [I32, I32, I32, I32, VP, P(I32), VP, VP, I32, VP]
        L.hs_indexer_topk_static.restype = ctypes.c_int
        L.hs_indexer_topk_static_error.argtypes = [I32, P(ctypes.c_uint32)]
        L.hs_indexer_topk_static_error.restype = ctypes.c_int
        _LIB = L
    return _LIB


def status_name(s: int) -> str:
    try:
        return lib().hs_status_string(s).decode()
    except OSError:
        return str(s)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def indexer_topk_static(idx_keys, lengths, q_idx, top_k: int, sel_out=None, stream=None):
    """Top-k selection with no device allocation inside the library (see
    hs_indexer_topk_static in include/hs.h).  idx_keys: int8 cuda [n_req, n_max,
    d_idx]; lengths: host ints [n_req]; q_idx: int8 cuda [n_req, d_idx]."""
    import torch
    n_req, n_max, d_idx = (int(x) for x in idx_keys.shape)
    if sel_out is None:
        sel_out = torch.empty((n_req, top_k), dtype=torch.int32, device=idx_keys.device)
    lens = (ctypes.c_int32 * max(1, n_req))(*[int(x) for x in lengths])
    rc = lib().hs_indexer_topk_static(n_req, n_max, d_idx, top_k, _ptr(idx_keys), lens, _ptr(q_idx),
                                      _ptr(sel_out), idx_keys.device.index or 0, _stream(stream))
    if rc != HS_OK:
        raise HsError(rc, lib().hs_last_error(None).decode())
    return sel_out


def indexer_topk_static_error(device: int = 0) -> int:
    """Device error word (HS_DEVERR_* bits) of the last indexer_topk_static call
    on `device` (synchronises the device)."""
    w = ctypes.c_uint32(0)
    rc = lib().hs_indexer_topk_static_error(device, ctypes.byref(w))
    if rc not in (HS_OK, HS_ERR_DEVICE):
        raise HsError(rc, lib().hs_last_error(None).decode())
    return int(w.value)


class HiSparseCache:
    """One two-level KV cache (all layers, up to max_requests requests) on one GPU."""

    def __init__(self, *, n_layers: int, max_requests: int, max_context: int, h_q: int, h_kv: int,
                 d_qk: int, d_v: int, d_idx: int, top_k: int, hot_slots: int, shared_kv: bool = False,
                 softmax_scale: float = 0.0, device: int = 0, fetch_mode: int = 2,
                 replacement: str = "lru", replacement_seed: int = 0, write_allocate: bool = False,
                 idx_heads: int = 1, index_share: int = 1, share_prefetch: bool = True, page_size: int = 1):
        if replacement not in REPLACEMENT:
            raise ValueError(f"replacement must be one of {sorted(REPLACEMENT)}")
        self.cfg = HsConfig(n_layers, max_requests, max_context, h_q, h_kv, d_qk, d_v, int(shared_kv),
                            d_idx, top_k, hot_slots, softmax_scale, device, fetch_mode,
                            REPLACEMENT[replacement], replacement_seed, int(write_allocate), int(idx_heads),
                            int(index_share), int(share_prefetch), int(page_size))
        # bytes of one request's indexer query (heads, then weights and padding)
        self.q_idx_row = d_idx if idx_heads <= 1 else idx_heads * d_idx + 16
        self._h = ctypes.c_void_p()
        rc = lib().hs_create(ctypes.byref(self.cfg), ctypes.byref(self._h))
        if rc != HS_OK:
            raise HsError(rc, lib().hs_last_error(None).decode())
        self.row_elems = int(lib().hs_row_elems(ctypes.byref(self.cfg)))
        self.device = device

    # -- lifetime --------------------------------------------------------------
    def close(self):
        if self._h:
            lib().hs_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def _check(self, rc: int):
        if rc != HS_OK:
            raise HsError(rc, lib().hs_last_error(self._h).decode())

    # -- the path -----------------------------------------------------------------
    def append(self, layer: int, kv_rows, idx_keys, req_ids=None, stream=None):
        """kv_rows: bf16 [n_req, n_tok, row_elems] (cuda or pinned cpu); idx_keys: int8 [n_req, n_tok, d_idx]."""
        n_req, n_tok = int(idx_keys.shape[0]), int(idx_keys.shape[1])
        assert kv_rows.shape[:2] == idx_keys.shape[:2] and kv_rows.shape[-1] == self.row_elems
        assert kv_rows.is_contiguous() and idx_keys.is_contiguous()
        assert kv_rows.element_size() == 2 and idx_keys.element_size() == 1
        self._check(lib().hs_append(self._h, layer, n_req, _ptr(req_ids), n_tok, _ptr(kv_rows),
                                    _ptr(idx_keys), _stream(stream)))

    def decode_layer(self, layer: int, q_idx, q, out=None, sel_out=None, req_ids=None, stream=None,
                     new_kv=None, new_keys=None):
        """q_idx: int8 [n_req, d_idx]; q: bf16 [n_req, h_q, d_qk] -> out bf16 [n_req, h_q, d_v].

        new_kv (bf16 [n_req, row_elems]) / new_keys (int8 [n_req, d_idx]): append one
        token per request first, inside the decode kernels."""
        import torch
        n_req = int(q_idx.shape[0])
        assert q_idx.is_cuda and q.is_cuda and q_idx.is_contiguous() and q.is_contiguous()
        assert q_idx.element_size() == 1 and q_idx.numel() == n_req * self.q_idx_row
        assert tuple(q.shape) == (n_req, self.cfg.h_q, self.cfg.d_qk) and q.element_size() == 2
        if out is None:
            out = torch.empty((n_req, self.cfg.h_q, self.cfg.d_v), dtype=torch.bfloat16, device=q.device)
        assert out.is_contiguous() and out.element_size() == 2
        if sel_out is not None:
            assert sel_out.dtype == torch.int32 and tuple(sel_out.shape) == (n_req, self.cfg.top_k)
        if new_kv is not None:
            assert new_keys is not None and new_kv.is_contiguous() and new_keys.is_contiguous()
            assert new_kv.numel() == n_req * self.row_elems and new_kv.element_size() == 2
            assert new_keys.numel() == n_req * self.cfg.d_idx and new_keys.element_size() == 1
        self._check(lib().hs_decode_layer(self._h, layer, n_req, _ptr(req_ids), _ptr(q_idx), _ptr(q),
                                          _ptr(out), _ptr(sel_out), _ptr(new_kv), _ptr(new_keys),
                                          _stream(stream)))
        return out

    # -- introspection ---------------------------------------------------------------
    def stats(self) -> dict:
        st = HsStats()
        rc = lib().hs_stats(self._h, ctypes.byref(st))
        if rc not in (HS_OK, HS_ERR_DEVICE):
            self._check(rc)
        return st.as_dict()

    def snapshot(self, req: int, layer: int, n_page: int):
        """(page[n_page], reverse[B], stamp[B], order[B], (length, step, hits, misses)) as numpy."""
        import numpy as np
        B = self.cfg.hot_slots
        page = np.empty(n_page, np.int32)
        rev = np.empty(B, np.int32)
        stamp = np.empty(B, np.int32)
        order = np.empty(B, np.int32)
        sc = np.empty(4, np.int64)
        self._check(lib().hs_snapshot(self._h, req, layer, page.ctypes.data, n_page, rev.ctypes.data,
                                      stamp.ctypes.data, order.ctypes.data, sc.ctypes.data))
        return page, rev, stamp, order, tuple(int(x) for x in sc)

    def reset_request(self, req: int, stream=None):
        self._check(lib().hs_reset_request(self._h, req, _stream(stream)))

    def set_timing(self, enable: bool):
        self._check(lib().hs_set_timing(self._h, int(enable)))

    def kernel_times(self) -> dict:
        ms = (ctypes.c_double * HS_K_COUNT)()
        n = (ctypes.c_int64 * HS_K_COUNT)()
        self._check(lib().hs_kernel_times(self._h, ms, n))
        return {KERNEL_NAMES[i]: (float(ms[i]), int(n[i])) for i in range(HS_K_COUNT)}
