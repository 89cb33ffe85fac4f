"""ctypes binding of libmla.so: argument marshalling only.

Every function here turns torch tensors into pointers and sizes, calls the C
entry point of the same name, and raises MLAError on a non-OK status.  No
attention arithmetic happens in Python; there is no fallback path: if the
library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
                4: "MLA_ERR_TIMEOUT", 5: "MLA_ERR_DEVICE_RANGE", 6: "MLA_ERR_WORKSPACE"}


class MLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()

c_void_p, c_int, c_int64, c_float, c_size_t, c_uint32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                                          ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32)

_SIGNATURES = {
    "mla_version": ([], c_int),
    "mla_last_error_string": ([], ctypes.c_char_p),
    "mla_status_string": ([c_int], ctypes.c_char_p),
    "mla_check_device_status": ([c_void_p, c_void_p, ctypes.POINTER(c_uint32)], c_int),
    "mla_set_spin_limit": ([c_uint32], None),
    "mla_set_tile_keys": ([c_int, c_int], None),
    "mla_debug_inject_stall": ([c_int], None),
    "mla_prefill_workspace_size": ([c_int, c_int], c_size_t),
    "mla_prefill": ([c_void_p, c_int64, c_int64, c_void_p, c_int64, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                     c_int64, c_int64, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p],
                    c_int),
    "mla_prefill_split_workspace_size": ([c_int, c_int], c_size_t),
    "mla_prefill_split": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                           c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p],
                          c_int),
    "mla_decode_workspace_size": ([c_int, c_int, c_int], c_size_t),
    "mla_decode": ([c_void_p, c_void_p, c_int64, c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_float, c_int,
                    c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "mla_decode_ex_workspace_size": ([c_int, c_int, c_int, c_int], c_size_t),
    "mla_decode_ex": ([c_void_p, c_int, c_void_p, c_int64, c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_float,
                       c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "mla_decode_fp8_workspace_size": ([c_int, c_int, c_int, c_int], c_size_t),
    "mla_decode_fp8": ([c_void_p, c_int, c_void_p, c_float, c_int64, c_int, c_void_p, c_int, c_void_p, c_int, c_int,
                        c_float, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "mla_decode_noalloc": ([c_void_p, c_void_p, c_int64, c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_float,
                            c_int, c_void_p, c_void_p, c_void_p], c_int),
    "mla_sparse_workspace_size": ([c_int, c_int], c_size_t),
    "mla_sparse": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                    c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "mla_prefill_varlen_workspace_size": ([c_int, c_int], c_size_t),
    "mla_prefill_varlen": ([c_void_p, c_int64, c_int64, c_void_p, c_int64, c_void_p, c_void_p, c_int, c_int, c_int,
                            c_int, c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                            c_void_p], c_int),
    "mla_absorb_q": ([c_void_p, c_int64, c_int64, c_void_p, c_int, c_int, c_void_p, c_int64, c_int64, c_void_p,
                      c_size_t, c_void_p], c_int),
    "mla_project_out": ([c_void_p, c_void_p, c_int, c_int, c_void_p, c_int64, c_int64, c_void_p, c_size_t,
                         c_void_p], c_int),
    "mla_rope_append_workspace_size": ([c_int], c_size_t),
    "mla_rope_append": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_void_p, c_int64, c_int,
                         c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "mla_merge_lse": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int, c_void_p],
                      c_int),
}


def lib():
    """Load libmla.so once (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libmla.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def exported_symbols():
    return sorted(_SIGNATURES)


def _check(status: int):
    if status != MLA_OK:
        msg = lib().mla_last_error_string().decode(errors="replace")
        raise MLAError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, device=None, contiguous: bool = True, shape=None):
    """Refuse (MLAError, status 1) a tensor the C ABI would misread: wrong dtype or device, a
    strided view where the call takes dense rows, or an unexpected shape."""
    if not isinstance(t, torch.Tensor):
        raise MLAError(1, f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise MLAError(1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise MLAError(1, f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise MLAError(1, f"{name} is on {t.device}, expected {device}")
    if contiguous and not t.is_contiguous():
        raise MLAError(1, f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise MLAError(1, f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ---------------------------------------------------------------------------
# workspace: caller-owned scratch, cached per device; first bytes = status word
# ---------------------------------------------------------------------------
_ws_cache = {}


def workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    key = (device.type, device.index)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def check_device_status(ws: Optional[torch.Tensor] = None, device=None, stream=None) -> int:
    """Read and clear the device status word; raise MLAError if a kernel reported a fault."""
    if ws is None:
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        ws = workspace(256, device)
    detail = c_uint32(0)
    s = lib().mla_check_device_status(_ptr(ws), _stream(stream), ctypes.byref(detail))
    _check(s)
    return detail.value


def set_spin_limit(limit: int):
    lib().mla_set_spin_limit(int(limit))


def set_tile_keys(prefill_keys: int = 0, decode_keys: int = 0):
    """128 or 64 keys per score tile of mla_prefill and of mla_decode; 0 keeps / restores the
    default of each (128 for both)."""
    lib().mla_set_tile_keys(int(prefill_keys), int(decode_keys))


def inject_stall(enable: bool):
    """Tests only: make every later launch wait on a barrier nothing arrives on."""
    lib().mla_debug_inject_stall(1 if enable else 0)


# ---------------------------------------------------------------------------
# the calls
# ---------------------------------------------------------------------------
def mla_prefill(q: torch.Tensor, kv: torch.Tensor, scale: float, causal: bool = True, q_pos0: int = 0,
                kv_pos0: int = 0, kv_valid: int = -1, prev_out: Optional[torch.Tensor] = None,
                prev_lse: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, dv: int = 512, ws: Optional[torch.Tensor] = None, stream=None):
    """Absorbed causal MLA prefill: q [T,H,576], kv [Tkv,576] -> out [T,H,dv], lse [H,T]."""
    _need(q, "q", torch.bfloat16, contiguous=False)    # rows may be strided (the ABI takes strides)
    _need(kv, "kv", torch.bfloat16, q.device, contiguous=False)
    T, H, dk = q.shape
    Tkv = kv.shape[0]
    if q.stride(2) != 1 or kv.stride(1) != 1:
        raise MLAError(1, "q and kv need contiguous last dimensions")
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, q.device, shape=(T, H, dv))
    _need(lse, "lse", torch.float32, q.device, shape=(H, T))
    if prev_out is not None:
        _need(prev_out, "prev_out", torch.bfloat16, q.device, shape=(T, H, dv))
    if prev_lse is not None:
        _need(prev_lse, "prev_lse", torch.float32, q.device, shape=(H, T))
    nbytes = lib().mla_prefill_workspace_size(T, H)
    ws = workspace(nbytes, q.device) if ws is None else ws
    s = lib().mla_prefill(_ptr(q), q.stride(0), q.stride(1), _ptr(kv), kv.stride(0), T, H, Tkv, dk, dv, float(scale),
                          int(bool(causal)), int(q_pos0), int(kv_pos0), int(kv_valid), _ptr(prev_out),
                          _ptr(prev_lse), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return out, lse


def mla_prefill_varlen(q, kv, cu_seqlens_q, cu_seqlens_kv, scale: float, causal: bool = True, prev_out=None,
                       prev_lse=None, out=None, lse=None, dv: int = 512, ws=None, stream=None):
    """Packed batch of sequences: q [total_q,H,576], kv [total_kv,576], cu_seqlens_* HOST int32 [batch+1].
    Query i of sequence b sees its keys j <= kv_len - q_len + i (causal).  Returns out, lse [H,total_q]."""
    _need(q, "q", torch.bfloat16, contiguous=False)
    _need(kv, "kv", torch.bfloat16, q.device, contiguous=False)
    if q.dim() != 3 or kv.dim() != 2 or q.stride(2) != 1 or kv.stride(1) != 1:
        raise MLAError(1, "q [total_q, H, 576] and kv [total_kv, 576] with contiguous last dimensions")
    cq = torch.as_tensor(cu_seqlens_q, dtype=torch.int32).cpu().contiguous()
    ck = torch.as_tensor(cu_seqlens_kv, dtype=torch.int32).cpu().contiguous()
    if cq.dim() != 1 or cq.shape != ck.shape or cq.numel() < 1:
        raise MLAError(1, "cu_seqlens_q and cu_seqlens_kv: host int32 [batch + 1]")
    batch = cq.numel() - 1
    Tq, H, dk = q.shape
    if int(cq[-1]) != Tq or int(ck[-1]) > kv.shape[0]:
        raise MLAError(1, "cu_seqlens must end at the packed lengths of q and kv")
    if out is None:
        out = torch.empty((Tq, H, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, q.device, shape=(Tq, H, dv))
    _need(lse, "lse", torch.float32, q.device, shape=(H, Tq))
    if prev_out is not None:
        _need(prev_out, "prev_out", torch.bfloat16, q.device, shape=(Tq, H, dv))
    if prev_lse is not None:
        _need(prev_lse, "prev_lse", torch.float32, q.device, shape=(H, Tq))
    nbytes = lib().mla_prefill_varlen_workspace_size(Tq, H)
    ws = workspace(nbytes, q.device) if ws is None else ws
    s = lib().mla_prefill_varlen(_ptr(q), q.stride(0), q.stride(1), _ptr(kv), kv.stride(0),
                                 ctypes.c_void_p(cq.data_ptr()), ctypes.c_void_p(ck.data_ptr()), batch, H, dk, dv,
                                 float(scale), int(bool(causal)), _ptr(prev_out), _ptr(prev_lse), _ptr(out),
                                 _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return out, lse


def mla_prefill_split(q_nope, q_pe, k_nope, k_pe, v, seq_len: torch.Tensor, head_num: int, kv_head_num: int,
                      qk_scale: float, mask_type: int = 1, prev_out=None, prev_lse=None, out=None, lse=None,
                      ws=None, stream=None):
    """Ascend split-layout prefill: returns out [Nq,H,128], lse [H,Nq]. seq_len is a HOST int32 tensor."""
    for name, t in (("q_nope", q_nope), ("q_pe", q_pe), ("k_nope", k_nope), ("k_pe", k_pe), ("v", v)):
        _need(t, name, torch.bfloat16, q_nope.device)
        if not t.is_contiguous():
            raise MLAError(1, f"{name} must be contiguous")
    sl = seq_len.to("cpu", torch.int32).contiguous()
    rows = 1 if sl.dim() == 1 else 2
    batch = sl.shape[-1]
    Nq, H = q_nope.shape[0], q_nope.shape[1]
    if out is None:
        out = torch.empty((Nq, H, 128), dtype=torch.bfloat16, device=q_nope.device)
    if lse is None:
        lse = torch.empty((H, Nq), dtype=torch.float32, device=q_nope.device)
    nbytes = lib().mla_prefill_split_workspace_size(Nq, H)
    ws = workspace(nbytes, q_nope.device) if ws is None else ws
    s = lib().mla_prefill_split(_ptr(q_nope), _ptr(q_pe), _ptr(k_nope), _ptr(k_pe), _ptr(v),
                                ctypes.c_void_p(sl.data_ptr()), rows, batch, int(head_num), int(kv_head_num),
                                float(qk_scale), int(mask_type), _ptr(prev_out), _ptr(prev_lse), _ptr(out), _ptr(lse),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return out, lse


def mla_decode(q, kv_cache, block_table, lens, scale: float, num_splits: int = 0, out=None, lse=None, ws=None,
               stream=None):
    """Paged absorbed decode: q [B,H,576], kv_cache [pages,page,576] -> out [B,H,512], lse [B,H]."""
    _need(q, "q", torch.bfloat16)
    _need(kv_cache, "kv_cache", torch.bfloat16, q.device)
    _need(block_table, "block_table", torch.int32, q.device)
    _need(lens, "lens", torch.int32, q.device)
    if q.dim() != 3 or kv_cache.dim() != 3 or block_table.dim() != 2:
        raise MLAError(1, "q [B,H,576], kv_cache [pages,page,576], block_table [B,max_pages] expected")
    B, H, _ = q.shape
    num_pages, page_size, _ = kv_cache.shape
    _need(lens, "lens", torch.int32, q.device, shape=(B,))
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, q.device, shape=(B, H, 512))
    _need(lse, "lse", torch.float32, q.device, shape=(B, H))
    nbytes = lib().mla_decode_workspace_size(B, H, int(num_splits))
    ws = workspace(nbytes, q.device) if ws is None else ws
    s = lib().mla_decode(_ptr(q), _ptr(kv_cache), num_pages, page_size, _ptr(block_table), block_table.shape[1],
                         _ptr(lens), B, H, float(scale), int(num_splits), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                         _stream(stream))
    _check(s)
    return out, lse


def mla_decode_ex(q, kv_cache, block_table, lens, scale: float, sinks=None, num_splits: int = 0, out=None,
                  lse=None, ws=None, stream=None):
    """Decode with q_per_req tokens per request (q [B,s,H,576]; token i sits at position lens[b]-s+i,
    causal among the request's tokens) and optional per-head sink logits sinks [H] (fp32).
    Returns out [B,s,H,512], lse [B,s,H]."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4 or q.shape[3] != 576:
        raise MLAError(1, "q must be [B, q_per_req, H, 576]")
    B, S, H, _ = q.shape
    dev = q.device
    _need(kv_cache, "kv_cache", torch.bfloat16, dev)
    if kv_cache.dim() != 3 or block_table.dim() != 2:
        raise MLAError(1, "kv_cache [pages,page,576], block_table [B,max_pages] expected")
    _need(block_table, "block_table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev, shape=(B,))
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, shape=(H,))
    num_pages, page_size, _ = kv_cache.shape
    if out is None:
        out = torch.empty((B, S, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, shape=(B, S, H, 512))
    _need(lse, "lse", torch.float32, dev, shape=(B, S, H))
    nbytes = lib().mla_decode_ex_workspace_size(B, S, H, int(num_splits))
    ws = workspace(nbytes, dev) if ws is None else ws
    s = lib().mla_decode_ex(_ptr(q), S, _ptr(kv_cache), num_pages, page_size, _ptr(block_table),
                            block_table.shape[1], _ptr(lens), B, H, float(scale), _ptr(sinks), int(num_splits),
                            _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return out, lse


def mla_decode_fp8(q, kv_cache_e4m3, kv_scale: float, block_table, lens, scale: float, sinks=None,
                   num_splits: int = 0, out=None, lse=None, ws=None, stream=None):
    """Decode over an e4m3 latent cache (torch.float8_e4m3fn [pages,page,576]; value = e4m3 x kv_scale).
    q bf16 [B,H,576] or [B,s,H,576].  Returns out, lse shaped like mla_decode / mla_decode_ex."""
    single = q.dim() == 3
    q4 = q.unsqueeze(1) if single else q
    _need(q4, "q", torch.bfloat16)
    if q4.dim() != 4 or q4.shape[3] != 576:
        raise MLAError(1, "q must be [B, H, 576] or [B, q_per_req, H, 576]")
    B, S, H, _ = q4.shape
    dev = q4.device
    if kv_cache_e4m3.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise MLAError(1, "kv_cache_e4m3 must be torch.float8_e4m3fn (or its bytes as uint8)")
    _need(kv_cache_e4m3, "kv_cache_e4m3", kv_cache_e4m3.dtype, dev)
    if kv_cache_e4m3.dim() != 3 or kv_cache_e4m3.shape[2] != 576 or block_table.dim() != 2:
        raise MLAError(1, "kv_cache_e4m3 [pages,page,576], block_table [B,max_pages] expected")
    _need(block_table, "block_table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev, shape=(B,))
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, shape=(H,))
    num_pages, page_size, _ = kv_cache_e4m3.shape
    if out is None:
        out = torch.empty((B, S, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    o4 = out.unsqueeze(1) if (single and out.dim() == 3) else out
    l3 = lse.unsqueeze(1) if (single and lse.dim() == 2) else lse
    _need(o4, "out", torch.bfloat16, dev, shape=(B, S, H, 512))
    _need(l3, "lse", torch.float32, dev, shape=(B, S, H))
    nbytes = lib().mla_decode_fp8_workspace_size(B, S, H, int(num_splits))
    ws = workspace(nbytes, dev) if ws is None else ws
    s = lib().mla_decode_fp8(_ptr(q4), S, _ptr(kv_cache_e4m3), float(kv_scale), num_pages, page_size,
                             _ptr(block_table), block_table.shape[1], _ptr(lens), B, H, float(scale), _ptr(sinks),
                             int(num_splits), _ptr(o4), _ptr(l3), _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return (o4[:, 0], l3[:, 0]) if single else (o4, l3)


def mla_decode_noalloc(q, kv_cache, block_table, lens, scale: float, num_splits: int = 0, out=None, lse=None,
                       stream=None):
    """mla_decode with its scratch in the library's fixed device array (no workspace, no allocation)."""
    _need(q, "q", torch.bfloat16)
    _need(kv_cache, "kv_cache", torch.bfloat16, q.device)
    _need(block_table, "block_table", torch.int32, q.device)
    _need(lens, "lens", torch.int32, q.device)
    if q.dim() != 3 or kv_cache.dim() != 3 or block_table.dim() != 2:
        raise MLAError(1, "q [B,H,576], kv_cache [pages,page,576], block_table [B,max_pages] expected")
    B, H, _ = q.shape
    num_pages, page_size, _ = kv_cache.shape
    _need(lens, "lens", torch.int32, q.device, shape=(B,))
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, q.device, shape=(B, H, 512))
    _need(lse, "lse", torch.float32, q.device, shape=(B, H))
    s = lib().mla_decode_noalloc(_ptr(q), _ptr(kv_cache), num_pages, page_size, _ptr(block_table),
                                 block_table.shape[1], _ptr(lens), B, H, float(scale), int(num_splits), _ptr(out),
                                 _ptr(lse), _stream(stream))
    _check(s)
    return out, lse


def mla_sparse(q_lift, q_pe, c_kv, k_pe, topk, softmax_scale: float, out=None, lse=None, ws=None, stream=None):
    """Top-k sparse MLA: returns out [B,S,H*512] (natural order), lse [B,S,H] (lse=False: no LSE is
    written and None is returned for it)."""
    for name, t in (("q_lift", q_lift), ("q_pe", q_pe), ("c_kv", c_kv), ("k_pe", k_pe)):
        _need(t, name, torch.bfloat16, q_lift.device)
    _need(topk, "topk", torch.int32, q_lift.device)
    if q_lift.dim() != 4 or c_kv.dim() != 3 or topk.dim() != 3:
        raise MLAError(1, "q_lift [B,S,H,512], c_kv [B,S_kv,512], topk [B,S,K] expected")
    B, S, H, L = q_lift.shape
    S_kv = c_kv.shape[1]
    K = topk.shape[-1]
    _need(q_pe, "q_pe", torch.bfloat16, q_lift.device, shape=(B, S, H, 64))
    _need(k_pe, "k_pe", torch.bfloat16, q_lift.device, shape=(B, S_kv, 64))
    _need(topk, "topk", torch.int32, q_lift.device, shape=(B, S, K))
    if out is None:
        out = torch.empty((B, S, H * L), dtype=torch.bfloat16, device=q_lift.device)
    no_lse = lse is False
    if lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=q_lift.device)
    _need(out, "out", torch.bfloat16, q_lift.device, shape=(B, S, H * L))
    if not no_lse:
        _need(lse, "lse", torch.float32, q_lift.device, shape=(B, S, H))
    nbytes = lib().mla_sparse_workspace_size(S, H)
    ws = workspace(nbytes, q_lift.device) if ws is None else ws
    s = lib().mla_sparse(_ptr(q_lift), _ptr(q_pe), _ptr(c_kv), _ptr(k_pe), _ptr(topk), B, S, S_kv, H, K,
                         float(softmax_scale), _ptr(out), None if no_lse else _ptr(lse), _ptr(ws), ws.numel(),
                         _stream(stream))
    _check(s)
    return out, (None if no_lse else lse)


def mla_absorb_q(q_nope, k_b_proj_trans, q_out=None, ws=None, stream=None):
    """q_out[t, h, :512] = q_nope[t, h] @ k_b_proj_trans[h].T.  q_nope [T,H,128] may be a strided view
    (last dimension contiguous); q_out defaults to a new fused query [T,H,576] (columns 512.. unset)."""
    _need(q_nope, "q_nope", torch.bfloat16, contiguous=False)
    if q_nope.dim() != 3 or q_nope.shape[2] != 128 or q_nope.stride(2) != 1:
        raise MLAError(1, "q_nope must be [T, H, 128] with a contiguous last dimension")
    T, H, _ = q_nope.shape
    dev = q_nope.device
    _need(k_b_proj_trans, "k_b_proj_trans", torch.bfloat16, dev, shape=(H, 512, 128))
    if q_out is None:
        q_out = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", torch.bfloat16, dev, contiguous=False)
    if q_out.dim() != 3 or q_out.shape[:2] != (T, H) or q_out.shape[2] < 512 or q_out.stride(2) != 1:
        raise MLAError(1, "q_out must be [T, H, >= 512] with a contiguous last dimension")
    ws = workspace(256, dev) if ws is None else ws
    s = lib().mla_absorb_q(_ptr(q_nope), q_nope.stride(0), q_nope.stride(1), _ptr(k_b_proj_trans), T, H,
                           _ptr(q_out), q_out.stride(0), q_out.stride(1), _ptr(ws), ws.numel(), _stream(stream))
    _check(s)
    return q_out


def mla_project_out(o_latent, v_b_proj, out=None, ws=None, stream=None):
    """out[t, h] = o_latent[t, h] @ v_b_proj[h].T: o_latent [T,H,512], v_b_proj [H,128,512] -> [T,H,128]."""
    _need(o_latent, "o_latent", torch.bfloat16)
    if o_latent.dim() != 3 or o_latent.shape[2] != 512:
        raise MLAError(1, "o_latent must be [T, H, 512]")
    T, H, _ = o_latent.shape
    dev = o_latent.device
    _need(v_b_proj, "v_b_proj", torch.bfloat16, dev, shape=(H, 128, 512))
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev, contiguous=False)
    if out.dim() != 3 or out.shape != (T, H, 128) or out.stride(2) != 1:
        raise MLAError(1, "out must be [T, H, 128] with a contiguous last dimension")
    ws = workspace(256, dev) if ws is None else ws
    s = lib().mla_project_out(_ptr(o_latent), _ptr(v_b_proj), T, H, _ptr(out), out.stride(0), out.stride(1), _ptr(ws),
                              ws.numel(), _stream(stream))
    _check(s)
    return out


def mla_rope_append(q_pe, c_kv, k_pe, positions, cos_sin, kv_cache, block_table, q_out, is_neox: bool = False,
                    ws=None, stream=None):
    """Decode step: rotate q_pe [B,H,64] into q_out[:, :, 512:] and append [c_kv | rotated k_pe] at
    row positions[b] of request b's pages in kv_cache (in place).  Returns q_out."""
    _need(q_pe, "q_pe", torch.bfloat16)
    if q_pe.dim() != 3 or q_pe.shape[2] != 64:
        raise MLAError(1, "q_pe must be [B, H, 64]")
    B, H, _ = q_pe.shape
    dev = q_pe.device
    _need(c_kv, "c_kv", torch.bfloat16, dev, shape=(B, 512))
    _need(k_pe, "k_pe", torch.bfloat16, dev, shape=(B, 64))
    _need(positions, "positions", torch.int32, dev, shape=(B,))
    _need(cos_sin, "cos_sin", torch.float32, dev)
    if cos_sin.dim() != 2 or cos_sin.shape[1] != 64:
        raise MLAError(1, "cos_sin must be [max_pos, 64]")
    _need(kv_cache, "kv_cache", torch.bfloat16, dev)
    if kv_cache.dim() != 3 or kv_cache.shape[2] != 576:
        raise MLAError(1, "kv_cache must be [pages, page_size, 576]")
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise MLAError(1, "block_table must be [B, max_pages]")
    _need(q_out, "q_out", torch.bfloat16, dev, shape=(B, H, 576))
    nbytes = lib().mla_rope_append_workspace_size(B)
    ws = workspace(nbytes, dev) if ws is None else ws
    s = lib().mla_rope_append(_ptr(q_pe), _ptr(c_kv), _ptr(k_pe), _ptr(positions), _ptr(cos_sin), cos_sin.shape[0],
                              int(bool(is_neox)), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1],
                              _ptr(block_table), block_table.shape[1], B, H, _ptr(q_out), _ptr(ws), ws.numel(),
                              _stream(stream))
    _check(s)
    return q_out


def mla_merge_lse(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None):
    """Merge two partial results by LSE: out_* [rows,H,dv] bf16, lse_* [H,rows] fp32."""
    _need(out_a, "out_a", torch.bfloat16)
    if out_a.dim() != 3:
        raise MLAError(1, "out_a must be [rows, H, dv]")
    rows, H, dv = out_a.shape
    dev = out_a.device
    _need(out_b, "out_b", torch.bfloat16, dev, shape=(rows, H, dv))
    _need(lse_a, "lse_a", torch.float32, dev, shape=(H, rows))
    _need(lse_b, "lse_b", torch.float32, dev, shape=(H, rows))
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    _need(out, "out", torch.bfloat16, dev, shape=(rows, H, dv))
    _need(lse, "lse", torch.float32, dev, shape=(H, rows))
    s = lib().mla_merge_lse(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out), _ptr(lse), rows, H, dv,
                            _stream(stream))
    _check(s)
    return out, lse
