"""Python binding of libpkv — paged-KV single-token decode attention on GB300.

Thin ctypes marshalling over the C ABI declared in include/pkv.h: the
functions below have the C names, take torch tensors (or raw integers for
pointers), pass their data pointers and the current CUDA stream, and turn a
negative status into an exception. Every step of the hot path runs in the
library's CUDA kernels; there is no fallback of any kind. Build the library
with ``python -c "import __graft_entry__ as g; g.build()"`` (or
``python paged_kv_decode_pagetable_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

# status codes (include/pkv.h)
PKV_OK = 0
PKV_E_NO_SLOT = -1
PKV_E_NO_PAGES = -2
PKV_E_BAD_SLOT = -3
PKV_E_BAD_ARG = -4
PKV_E_CUDA = -5
# device error-word bits
PKV_ERR_POS = 1
PKV_ERR_PAGE_RANGE = 2
PKV_ERR_PAGE_NEG = 4
PKV_ERR_SLOT = 8
PKV_ERR_TIMEOUT = 16


class PkvError(RuntimeError):
    code = None


class NoSlotError(PkvError):
    code = PKV_E_NO_SLOT


class NoPagesError(PkvError):
    code = PKV_E_NO_PAGES


class BadSlotError(PkvError):
    code = PKV_E_BAD_SLOT


class BadArgError(PkvError):
    code = PKV_E_BAD_ARG


class CudaError(PkvError):
    code = PKV_E_CUDA


_ERRORS = {c.code: c for c in (NoSlotError, NoPagesError, BadSlotError, BadArgError, CudaError)}

_c_int, _c_p, _c_f, _c_sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
_c_ip = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "pt_create": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_p, _c_p, ctypes.POINTER(_c_p)]),
    "pt_destroy": (_c_int, [_c_p]),
    "pt_set_stream": (_c_int, [_c_p, _c_p]),
    "pt_can_reserve": (_c_int, [_c_p, _c_int, _c_int, ctypes.POINTER(_c_int)]),
    "pt_assign": (_c_int, [_c_p, _c_int, ctypes.POINTER(_c_int)]),
    "pt_reserve": (_c_int, [_c_p, _c_int, _c_int]),
    "pt_free": (_c_int, [_c_p, _c_int]),
    "pt_capacity": (_c_int, [_c_p, _c_int, ctypes.POINTER(_c_int)]),
    "pt_pages": (_c_int, [_c_p, _c_int, _c_ip, _c_int, ctypes.POINTER(_c_int)]),
    "pt_free_pages": (_c_int, [_c_p, ctypes.POINTER(_c_int)]),
    "pt_free_page_list": (_c_int, [_c_p, _c_ip, _c_int, ctypes.POINTER(_c_int)]),
    "pt_host_table": (_c_int, [_c_p, _c_ip, _c_int]),
    "kv_append": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_int, _c_int, _c_int,
                           _c_int, _c_p, _c_p, _c_int, _c_int, _c_p, _c_p]),
    "kv_append_prefill": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_int, _c_int, _c_int,
                                   _c_int, _c_p, _c_p, _c_int, _c_int, _c_p, _c_p]),
    "prefill_block_mask": (_c_int, [_c_p, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "convert_logical_block_mask": (_c_int, [_c_p, _c_int, _c_int, _c_p, _c_int, _c_int, _c_int,
                                            _c_int, _c_p, _c_int, _c_p, _c_p, _c_p]),
    "prefill_attn": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int,
                              _c_int, _c_int, _c_int, _c_f, _c_p, _c_p]),
    "qk_norm_rope": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_f, _c_int, _c_int,
                              _c_int, _c_int, _c_p]),
    "qk_norm_rope_append": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_f,
                                     _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_int,
                                     _c_int, _c_int, _c_p, _c_p, _c_p, _c_p]),
    "paged_decode_attn": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int,
                                   _c_p, _c_p, _c_int, _c_f, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_p, _c_sz, _c_p, _c_p, _c_p]),
    "paged_decode_attn_noalloc": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int,
                                           _c_int, _c_p, _c_p, _c_int, _c_f, _c_int, _c_int,
                                           _c_int, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "paged_decode_attn_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          ctypes.POINTER(_c_int)]),
    "paged_decode_attn_workspace": (_c_sz, [_c_int, _c_int, _c_int, _c_int]),
    "qkv_norm_rope": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_f, _c_int, _c_int,
                               _c_int, _c_int, _c_int, _c_p]),
    "paged_decode_step_ex": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_f,
                                      _c_int, _c_int, _c_int, _c_p, _c_int, _c_int, _c_int,
                                      _c_int, _c_p, _c_p, _c_int, _c_f, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_p, _c_sz, _c_p, _c_p, _c_p]),
    "paged_decode_step": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_f, _c_p,
                                   _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_int, _c_f,
                                   _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_sz, _c_p,
                                   _c_p, _c_p]),
    "pkv_read_error_word": (_c_int, [_c_p, _c_p, _c_ip]),
    "pkv_last_error": (ctypes.c_char_p, []),
}

EXPORTS = tuple(_SIGS)
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libpkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libpkv.so not found at {path}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        msg = load_library().pkv_last_error().decode(errors="replace")
        raise _ERRORS.get(status, PkvError)(f"{what}: {msg} (status {status})")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _bf16(t, name):
    if t is not None and not isinstance(t, int):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise BadArgError(f"{name} must be a contiguous bfloat16 tensor")
    return t


def _i32(t, name):
    if t is not None and not isinstance(t, int):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise BadArgError(f"{name} must be a contiguous int32 tensor")
    return t


# --------------------------------------------------------------------------
# PageTable allocator
# --------------------------------------------------------------------------

def pt_create(max_batch_size: int, page_size: int, n_pages: int, max_pages_per_seq: int,
              dev_table=None, stream=None) -> int:
    lib = load_library()
    h = _c_p()
    _check(lib.pt_create(max_batch_size, page_size, n_pages, max_pages_per_seq,
                         _ptr(_i32(dev_table, "dev_table")), _stream(stream) if dev_table is not None else None,
                         ctypes.byref(h)), "pt_create")
    return h.value


def pt_destroy(h: int) -> None:
    _check(load_library().pt_destroy(h), "pt_destroy")


def pt_set_stream(h: int, stream=None) -> None:
    _check(load_library().pt_set_stream(h, _stream(stream)), "pt_set_stream")


def pt_can_reserve(h: int, seq_len: int, slot: int = -1) -> bool:
    ok = _c_int()
    _check(load_library().pt_can_reserve(h, seq_len, slot, ctypes.byref(ok)), "pt_can_reserve")
    return bool(ok.value)


def pt_assign(h: int, seq_len: int) -> int:
    slot = _c_int()
    _check(load_library().pt_assign(h, seq_len, ctypes.byref(slot)), "pt_assign")
    return slot.value


def pt_reserve(h: int, slot: int, seq_len: int) -> None:
    _check(load_library().pt_reserve(h, slot, seq_len), "pt_reserve")


def pt_free(h: int, slot: int) -> None:
    _check(load_library().pt_free(h, slot), "pt_free")


def pt_capacity(h: int, slot: int) -> int:
    n = _c_int()
    _check(load_library().pt_capacity(h, slot, ctypes.byref(n)), "pt_capacity")
    return n.value


def pt_pages(h: int, slot: int) -> list[int]:
    lib = load_library()
    n = _c_int()
    _check(lib.pt_pages(h, slot, None, 0, ctypes.byref(n)), "pt_pages")
    buf = (ctypes.c_int32 * max(n.value, 1))()
    _check(lib.pt_pages(h, slot, buf, n.value, ctypes.byref(n)), "pt_pages")
    return list(buf[:n.value])


def pt_free_pages(h: int) -> int:
    n = _c_int()
    _check(load_library().pt_free_pages(h, ctypes.byref(n)), "pt_free_pages")
    return n.value


def pt_free_page_list(h: int) -> list[int]:
    lib = load_library()
    n = _c_int()
    _check(lib.pt_free_page_list(h, None, 0, ctypes.byref(n)), "pt_free_page_list")
    buf = (ctypes.c_int32 * max(n.value, 1))()
    _check(lib.pt_free_page_list(h, buf, n.value, ctypes.byref(n)), "pt_free_page_list")
    return list(buf[:n.value])


def pt_host_table(h: int, n_slots: int, max_pages_per_seq: int) -> torch.Tensor:
    out = torch.empty((n_slots, max_pages_per_seq), dtype=torch.int32)
    _check(load_library().pt_host_table(h, ctypes.cast(out.data_ptr(), _c_ip), out.numel()),
           "pt_host_table")
    return out


class PageTable:
    """Owns one pt_* handle and its caller-side device table tensor."""

    def __init__(self, max_batch_size: int, page_size: int, n_pages: int,
                 max_pages_per_seq: int, device=None, stream=None):
        self.max_batch_size = max_batch_size
        self.n_slots = max_batch_size + 1
        self.page_size = page_size
        self.n_pages = n_pages
        self.max_pages_per_seq = max_pages_per_seq
        self.dev_table = None
        if device is not None:
            self.dev_table = torch.empty((self.n_slots, max_pages_per_seq),
                                         dtype=torch.int32, device=device)
        self.handle = pt_create(max_batch_size, page_size, n_pages, max_pages_per_seq,
                                self.dev_table, stream)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.pt_destroy(h)
            self.handle = None

    def can_reserve(self, seq_len, slot=-1):
        return pt_can_reserve(self.handle, seq_len, slot)

    def assign(self, seq_len):
        return pt_assign(self.handle, seq_len)

    def reserve(self, slot, seq_len):
        pt_reserve(self.handle, slot, seq_len)

    def free(self, slot):
        pt_free(self.handle, slot)

    def capacity(self, slot):
        return pt_capacity(self.handle, slot)

    def pages(self, slot):
        return pt_pages(self.handle, slot)

    def free_page_list(self):
        return pt_free_page_list(self.handle)

    def host_table(self):
        return pt_host_table(self.handle, self.n_slots, self.max_pages_per_seq)


# --------------------------------------------------------------------------
# kernels
# --------------------------------------------------------------------------

def kv_append(k, v, batch_idx, input_pos, dev_table, n_slots, max_pages_per_seq,
              page_size, n_pages, k_cache, v_cache, err_word=None, stream=None) -> None:
    _bf16(k, "k"), _bf16(v, "v"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(batch_idx, "batch_idx"), _i32(input_pos, "input_pos"), _i32(dev_table, "dev_table")
    B, Hkv, D = k.shape
    _check(load_library().kv_append(
        _ptr(k), _ptr(v), _ptr(batch_idx), _ptr(input_pos), B, _ptr(dev_table), n_slots,
        max_pages_per_seq, page_size, n_pages, _ptr(k_cache), _ptr(v_cache), Hkv, D,
        _ptr(err_word), _stream(stream)), "kv_append")


def kv_append_prefill(k, v, batch_idx, input_pos, dev_table, n_slots, max_pages_per_seq,
                      page_size, n_pages, k_cache, v_cache, err_word=None, stream=None) -> None:
    """Scatter L packed prefill tokens; k and v are head-major [Hkv][L][D]."""
    _bf16(k, "k"), _bf16(v, "v"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(batch_idx, "batch_idx"), _i32(input_pos, "input_pos"), _i32(dev_table, "dev_table")
    Hkv, L, D = k.shape
    _check(load_library().kv_append_prefill(
        _ptr(k), _ptr(v), _ptr(batch_idx), _ptr(input_pos), L, _ptr(dev_table), n_slots,
        max_pages_per_seq, page_size, n_pages, _ptr(k_cache), _ptr(v_cache), Hkv, D,
        _ptr(err_word), _stream(stream)), "kv_append_prefill")


def qk_norm_rope(q, k, gamma_q, gamma_k, pos, theta: float, eps: float = 1e-6,
                 stream=None) -> None:
    _bf16(q, "q"), _bf16(k, "k"), _bf16(gamma_q, "gamma_q"), _bf16(gamma_k, "gamma_k")
    _i32(pos, "pos")
    B, Hq, D = q.shape
    Hkv = 0 if k is None else k.shape[1]
    _check(load_library().qk_norm_rope(
        _ptr(q), _ptr(k), _ptr(gamma_q), _ptr(gamma_k), _ptr(pos), float(theta), float(eps),
        B, Hq, Hkv, D, _stream(stream)), "qk_norm_rope")


def qkv_norm_rope(q, k, v, gamma_q, gamma_k, pos, theta: float, eps: float = 1e-6,
                  rotary_dims: int | None = None, stream=None) -> None:
    """qk_norm_rope with partial rotary (leading rotary_dims of D) and, when v
    is given, v normalised in place without a gain."""
    _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(gamma_q, "gamma_q")
    _bf16(gamma_k, "gamma_k"), _i32(pos, "pos")
    B, Hq, D = q.shape
    Hkv = 0 if k is None else k.shape[1]
    rd = D if rotary_dims is None else int(rotary_dims)
    _check(load_library().qkv_norm_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _ptr(pos), float(theta),
        float(eps), rd, B, Hq, Hkv, D, _stream(stream)), "qkv_norm_rope")


def qk_norm_rope_append(q, k, v, gamma_q, gamma_k, batch_idx, input_pos, theta: float,
                        eps, dev_table, n_slots, max_pages_per_seq, page_size, n_pages,
                        k_cache, v_cache, err_word=None, stream=None) -> None:
    _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(gamma_q, "gamma_q")
    _bf16(gamma_k, "gamma_k"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(batch_idx, "batch_idx"), _i32(input_pos, "input_pos"), _i32(dev_table, "dev_table")
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    _check(load_library().qk_norm_rope_append(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _ptr(batch_idx),
        _ptr(input_pos), float(theta), float(eps), B, Hq, Hkv, D, _ptr(dev_table), n_slots,
        max_pages_per_seq, page_size, n_pages, _ptr(k_cache), _ptr(v_cache), _ptr(err_word),
        _stream(stream)), "qk_norm_rope_append")


def paged_decode_attn_splits(B, Hkv, D, max_pages_per_seq, page_size, window=0) -> int:
    n = _c_int()
    _check(load_library().paged_decode_attn_splits(B, Hkv, D, max_pages_per_seq, page_size,
                                                   window, ctypes.byref(n)),
           "paged_decode_attn_splits")
    return n.value


def paged_decode_attn_workspace(B, Hq, D, num_splits) -> int:
    return int(load_library().paged_decode_attn_workspace(B, Hq, D, num_splits))


def paged_decode_attn(q, k_cache, v_cache, dev_table, n_slots, max_pages_per_seq, page_size,
                      n_pages, batch_idx, seq_lens, window, scale, num_splits, workspace,
                      out, err_word=None, stream=None) -> None:
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _bf16(out, "out")
    _i32(dev_table, "dev_table"), _i32(batch_idx, "batch_idx"), _i32(seq_lens, "seq_lens")
    B, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(dev_table), n_slots, max_pages_per_seq,
        page_size, n_pages, _ptr(batch_idx), _ptr(seq_lens), int(window), float(scale), B, Hq,
        Hkv, D, int(num_splits), _ptr(workspace), ws_bytes, _ptr(out), _ptr(err_word),
        _stream(stream)), "paged_decode_attn")


def paged_decode_step(q, k, v, gamma_q, gamma_k, batch_idx, input_pos, theta, eps, dev_table,
                      n_slots, max_pages_per_seq, page_size, n_pages, k_cache, v_cache, window,
                      scale, num_splits, workspace, out, err_word=None, stream=None) -> None:
    """qk_norm_rope + kv_append + paged_decode_attn (seq_lens = input_pos + 1)
    in one pass; q, k and v are read only."""
    _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(gamma_q, "gamma_q")
    _bf16(gamma_k, "gamma_k"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _bf16(out, "out")
    _i32(dev_table, "dev_table"), _i32(batch_idx, "batch_idx"), _i32(input_pos, "input_pos")
    B, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().paged_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _ptr(batch_idx),
        _ptr(input_pos), float(theta), float(eps), _ptr(dev_table), n_slots, max_pages_per_seq,
        page_size, n_pages, _ptr(k_cache), _ptr(v_cache), int(window), float(scale), B, Hq, Hkv,
        D, int(num_splits), _ptr(workspace), ws_bytes, _ptr(out), _ptr(err_word),
        _stream(stream)), "paged_decode_step")


def paged_decode_step_ex(q, k, v, gamma_q, gamma_k, batch_idx, input_pos, theta, eps,
                         rotary_dims, v_norm, k_eq_v, dev_table, n_slots, max_pages_per_seq,
                         page_size, n_pages, k_cache, v_cache, window, scale, num_splits,
                         workspace, out, err_word=None, stream=None) -> None:
    """paged_decode_step with the Gemma-4 options: rotary on the leading
    rotary_dims (None: all of D), gain-free value norm, value = raw k."""
    _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(gamma_q, "gamma_q")
    _bf16(gamma_k, "gamma_k"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _bf16(out, "out")
    _i32(dev_table, "dev_table"), _i32(batch_idx, "batch_idx"), _i32(input_pos, "input_pos")
    B, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    rd = D if rotary_dims is None else int(rotary_dims)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().paged_decode_step_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma_q), _ptr(gamma_k), _ptr(batch_idx),
        _ptr(input_pos), float(theta), float(eps), rd, int(bool(v_norm)), int(bool(k_eq_v)),
        _ptr(dev_table), n_slots, max_pages_per_seq, page_size, n_pages, _ptr(k_cache),
        _ptr(v_cache), int(window), float(scale), B, Hq, Hkv, D, int(num_splits),
        _ptr(workspace), ws_bytes, _ptr(out), _ptr(err_word), _stream(stream)),
        "paged_decode_step_ex")


def paged_decode_attn_noalloc(q, k_cache, v_cache, dev_table, n_slots, max_pages_per_seq,
                              page_size, n_pages, batch_idx, seq_lens, window, scale, num_splits,
                              out, err_word=None, stream=None) -> None:
    """paged_decode_attn for callers that cannot allocate device memory: the
    split partials go to the library's fixed 32 MiB device scratch instead
    of a caller workspace. Calls share that scratch, so calls that overlap on
    the GPU must be serialized by the caller."""
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _bf16(out, "out")
    _i32(dev_table, "dev_table"), _i32(batch_idx, "batch_idx"), _i32(seq_lens, "seq_lens")
    B, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    _check(load_library().paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(dev_table), n_slots, max_pages_per_seq,
        page_size, n_pages, _ptr(batch_idx), _ptr(seq_lens), int(window), float(scale), B, Hq,
        Hkv, D, int(num_splits), _ptr(out), _ptr(err_word), _stream(stream)),
        "paged_decode_attn_noalloc")


def convert_logical_block_mask(kv_indices, dev_table, n_slots, max_pages_per_seq,
                               batch_idx=None, n_cols=None, err_word=None, stream=None):
    """Logical -> physical key-block indices of a block mask (int32
    [B][H][rows][max_blocks], device) through the page table; returns int32
    [B][H][rows][n_cols] (n_cols defaults to max(max_blocks, max_pages_per_seq))."""
    _i32(kv_indices, "kv_indices"), _i32(dev_table, "dev_table"), _i32(batch_idx, "batch_idx")
    if kv_indices.dim() != 4:
        raise BadArgError("kv_indices must be [B][H][rows][max_blocks]")
    B, H, R, M = kv_indices.shape
    if n_cols is None:
        n_cols = max(M, max_pages_per_seq)
    out = torch.empty((B, H, R, n_cols), dtype=torch.int32, device=kv_indices.device)
    _check(load_library().convert_logical_block_mask(
        _ptr(dev_table), n_slots, max_pages_per_seq, _ptr(batch_idx), B, H, R, M,
        _ptr(kv_indices), n_cols, _ptr(out), _ptr(err_word), _stream(stream)),
        "convert_logical_block_mask")
    return out


PREFILL_BLOCK = 64


class PrefillBlockMask:
    """The block mask prefill_block_mask writes (int32 device tensors):
    kv_num_blocks [n], kv_indices [n][n] (partial blocks),
    full_kv_num_blocks [n], full_kv_indices [n][n], for n = ceil(L / 64),
    plus the docs and window it was built for."""

    __slots__ = ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices",
                 "docs", "window")

    def __init__(self, kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices, docs,
                 window):
        self.kv_num_blocks = kv_num_blocks
        self.kv_indices = kv_indices
        self.full_kv_num_blocks = full_kv_num_blocks
        self.full_kv_indices = full_kv_indices
        self.docs = docs
        self.window = int(window)


def prefill_block_mask(docs, window: int = 0, stream=None) -> PrefillBlockMask:
    """Builds the document-causal (window > 0: sliding) block mask of the
    packed tokens' document ids docs (int32 [L], device)."""
    _i32(docs, "docs")
    L = docs.numel()
    n = -(-L // PREFILL_BLOCK)
    dev = docs.device
    bm = PrefillBlockMask(torch.empty(n, dtype=torch.int32, device=dev),
                          torch.empty((n, n), dtype=torch.int32, device=dev),
                          torch.empty(n, dtype=torch.int32, device=dev),
                          torch.empty((n, n), dtype=torch.int32, device=dev), docs, window)
    _check(load_library().prefill_block_mask(
        _ptr(docs), L, int(window), _ptr(bm.kv_num_blocks), _ptr(bm.kv_indices),
        _ptr(bm.full_kv_num_blocks), _ptr(bm.full_kv_indices), _stream(stream)),
        "prefill_block_mask")
    return bm


def prefill_attn(q, k, v, block_mask: PrefillBlockMask, scale, out, stream=None) -> None:
    """Document-causal attention over packed tokens: q [Hq][L][D], k/v
    [Hkv][L][D], out [Hq][L][D]; block_mask from prefill_block_mask (its docs
    and window are the mask's)."""
    _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(out, "out")
    bm = block_mask
    for name in ("docs", "kv_num_blocks", "kv_indices", "full_kv_num_blocks",
                 "full_kv_indices"):
        _i32(getattr(bm, name), name)
    Hq, L, D = q.shape
    Hkv = k.shape[0]
    if bm.docs.numel() != L or bm.kv_num_blocks.numel() != -(-L // PREFILL_BLOCK):
        raise BadArgError("prefill_attn: block mask built for another length")
    _check(load_library().prefill_attn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(bm.docs), _ptr(bm.kv_num_blocks), _ptr(bm.kv_indices),
        _ptr(bm.full_kv_num_blocks), _ptr(bm.full_kv_indices), L, Hq, Hkv, D, bm.window,
        float(scale), _ptr(out), _stream(stream)), "prefill_attn")


def pkv_read_error_word(err_word, stream=None) -> int:
    v = ctypes.c_int32()
    _check(load_library().pkv_read_error_word(_ptr(err_word), _stream(stream), ctypes.byref(v)),
           "pkv_read_error_word")
    return v.value


def pkv_last_error() -> str:
    return load_library().pkv_last_error().decode(errors="replace")
