"""ctypes binding of libbsxattn.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; this module turns torch
tensors into device pointers, sizes and the current CUDA stream, calls the C
entry point of the same name and raises on a non-zero status.  There is no
other implementation to fall back to: if the shared library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsxattn.so")

BSX_F32, BSX_BF16, BSX_F8E4M3 = 0, 1, 2
BSX_FORCE_FIRST_LAST = 1
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "CUDA error",
          -4: "bounded device wait expired", -5: "workspace missing or too small"}

EXPORTS = ("bsx_version", "bsx_status_string", "bsx_estimate_workspace_bytes",
           "bsx_xattn_estimate", "bsx_bsa_prefill", "bsx_merge_attn",
           "bsx_map_mask_to_cpu_blocks", "bsx_last_error", "bsx_last_error_code",
           "bsx_xattn_estimate_noalloc",
           "bsx_cpu_block_mask", "bsx_chunk_prefill", "bsx_bsa_prefill_split",
           "bsx_quantize_e4m3", "bsx_chunk_step_host", "bsx_debug_drop_ring_item",
           "bsx_chunk_prefill_workspace_bytes", "bsx_debug_fused_skip_row", "bsx_chunk_step")
BSX_STEP_OFFLOAD, BSX_STEP_E4M3_ESTIMATE, BSX_STEP_FUSED = 2, 4, 8


class BsxShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("d", ctypes.c_int), ("dtype", ctypes.c_int)]


class BsxChunkBuffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("q", "k", "v", "mask", "bsa_mask", "o", "lse", "o_curr", "lse_curr", "keep",
                 "q8", "k8", "workspace")] + [("workspace_bytes", ctypes.c_size_t),
                                              ("done", ctypes.c_void_p)]


class BsxError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libbsxattn.so not found at {path}: build it with "
                "`python -m block_sparse_long_xattn_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.bsx_version.restype = i32
        lib.bsx_version.argtypes = []
        lib.bsx_status_string.restype = ctypes.c_char_p
        lib.bsx_status_string.argtypes = [i32]
        lib.bsx_estimate_workspace_bytes.restype = sz
        lib.bsx_estimate_workspace_bytes.argtypes = [BsxShape, i32, i32, i32]
        lib.bsx_xattn_estimate.restype = i32
        lib.bsx_xattn_estimate.argtypes = [BsxShape, vp, vp, i32, i32, i32, f32, vp, vp,
                                           vp, sz, vp]
        lib.bsx_xattn_estimate_noalloc.restype = i32
        lib.bsx_xattn_estimate_noalloc.argtypes = [BsxShape, vp, vp, i32, i32, i32, f32,
                                                   vp, vp, vp]
        lib.bsx_bsa_prefill.restype = i32
        lib.bsx_bsa_prefill.argtypes = [BsxShape, vp, vp, vp, vp, i32, i32, i32, i32,
                                        vp, vp, vp]
        lib.bsx_quantize_e4m3.restype = i32
        lib.bsx_quantize_e4m3.argtypes = [vp, vp, ctypes.c_longlong, vp]
        lib.bsx_bsa_prefill_split.restype = i32
        lib.bsx_bsa_prefill_split.argtypes = [BsxShape, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp,
                                              vp]
        lib.bsx_merge_attn.restype = i32
        lib.bsx_merge_attn.argtypes = [BsxShape, i32, vp, vp, vp, vp, vp]
        lib.bsx_map_mask_to_cpu_blocks.restype = i32
        lib.bsx_map_mask_to_cpu_blocks.argtypes = [BsxShape, vp, i32, i32, i32, i32, vp, vp]
        lib.bsx_chunk_step.restype = i32
        lib.bsx_chunk_step.argtypes = [BsxShape, vp, vp, vp, i32, i32, i32, f32, i32, vp, vp, vp,
                                       vp, vp, vp, vp, sz, vp]
        lib.bsx_chunk_prefill_workspace_bytes.restype = sz
        lib.bsx_chunk_prefill_workspace_bytes.argtypes = [BsxShape, i32, i32, i32]
        lib.bsx_chunk_prefill.restype = i32
        lib.bsx_chunk_prefill.argtypes = [BsxShape, vp, vp, vp, i32, i32, i32, f32, vp, vp,
                                          vp, vp, sz, vp]
        lib.bsx_cpu_block_mask.restype = i32
        lib.bsx_cpu_block_mask.argtypes = [BsxShape, vp, i32, i32, i32, vp, vp]
        lib.bsx_last_error.restype = i32
        lib.bsx_last_error.argtypes = [vp]
        lib.bsx_last_error_code.restype = ctypes.c_uint
        lib.bsx_last_error_code.argtypes = []
        lib.bsx_debug_fused_skip_row.restype = i32
        lib.bsx_debug_fused_skip_row.argtypes = [i32]
        lib.bsx_debug_drop_ring_item.restype = i32
        lib.bsx_debug_drop_ring_item.argtypes = [i32, i32]
        lib.bsx_chunk_step_host.restype = i32
        lib.bsx_chunk_step_host.argtypes = [BsxShape, vp, vp, vp, i32, i32, i32, f32, i32, i32,
                                            ctypes.POINTER(BsxChunkBuffers), vp, vp, vp, vp, vp,
                                            vp]
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise BsxError(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BSX_BF16
    if t.dtype == torch.float32:
        return BSX_F32
    if t.dtype == torch.float8_e4m3fn:
        return BSX_F8E4M3
    raise TypeError(f"unsupported dtype {t.dtype}; bsxattn takes bfloat16, float32 "
                    "or (estimate only) float8_e4m3fn")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("bsxattn takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("bsxattn takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("this argument is a host buffer")
    if not t.is_contiguous():
        raise ValueError("bsxattn takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def shape_of(q: torch.Tensor, k: torch.Tensor) -> BsxShape:
    B, _, Hq, d = q.shape
    Hkv = k.shape[2]
    return BsxShape(B, Hq, Hkv, d, _dtype_code(q))


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------
def bsx_version() -> int:
    return load().bsx_version()


def bsx_estimate_workspace_bytes(shape: BsxShape, q_len: int, q_start_pos: int,
                                 stride: int) -> int:
    return int(load().bsx_estimate_workspace_bytes(shape, q_len, q_start_pos, stride))


def bsx_xattn_estimate(q, k, q_start_pos: int, stride: int, threshold: float, *,
                       mask=None, block_sums=None, workspace=None, stream=None):
    """uint8 block mask [B, Hq, q_len/128, Lk/128] for the chunk (see bsxattn.h)."""
    lib = load()
    B, q_len, Hq, _ = q.shape
    Lk = k.shape[1]
    shape = shape_of(q, k)
    if mask is None:
        mask = torch.empty((B, Hq, q_len // 128, Lk // 128), dtype=torch.uint8, device=q.device)
    need = lib.bsx_estimate_workspace_bytes(shape, q_len, q_start_pos, stride)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("bsx_xattn_estimate", lib.bsx_xattn_estimate(
        shape, _ptr(q), _ptr(k), q_len, q_start_pos, stride, float(threshold),
        _ptr(mask), _ptr(block_sums), _ptr(workspace), ws_bytes, _stream(stream)))
    return mask


def bsx_xattn_estimate_noalloc(q, k, q_start_pos: int, stride: int, threshold: float,
                               *, mask, block_sums=None, stream=None):
    """bsx_xattn_estimate using the library's own scratch (no workspace, no
    allocation by the library or by this wrapper: `mask` must be provided)."""
    lib = load()
    _, q_len, _, _ = q.shape
    _check("bsx_xattn_estimate_noalloc", lib.bsx_xattn_estimate_noalloc(
        shape_of(q, k), _ptr(q), _ptr(k), q_len, q_start_pos, stride, float(threshold),
        _ptr(mask), _ptr(block_sums), _stream(stream)))
    return mask


def bsx_bsa_prefill(q, k, v, mask, q_start_pos: int, kb_begin: int = 0,
                    kb_end: int | None = None, *, o=None, lse=None, stream=None):
    """Block-sparse causal attention over key blocks [kb_begin, kb_end) -> (o, lse)."""
    lib = load()
    B, q_len, Hq, d = q.shape
    if kb_end is None:
        kb_end = k.shape[1] // 128
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, q_len), dtype=torch.float32, device=q.device)
    _check("bsx_bsa_prefill", lib.bsx_bsa_prefill(
        shape_of(q, k), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), q_len, q_start_pos,
        kb_begin, kb_end, _ptr(o), _ptr(lse), _stream(stream)))
    return o, lse


def bsx_quantize_e4m3(src, *, out=None, stream=None):
    """bf16 tensor -> float8_e4m3fn tensor of the same shape (nearest, ties to
    even, saturated to +-448)."""
    lib = load()
    if src.dtype != torch.bfloat16:
        raise TypeError("bsx_quantize_e4m3 takes bfloat16")
    if out is None:
        out = torch.empty(src.shape, dtype=torch.float8_e4m3fn, device=src.device)
    _check("bsx_quantize_e4m3", lib.bsx_quantize_e4m3(_ptr(src), _ptr(out), src.numel(),
                                                       _stream(stream)))
    return out


def bsx_bsa_prefill_split(q, k, v, mask, q_start_pos: int, *, o_hist=None, lse_hist=None,
                          o_curr=None, lse_curr=None, stream=None):
    """History and current-chunk block-sparse attention in one launch
    -> (o_hist, lse_hist, o_curr, lse_curr)."""
    lib = load()
    B, q_len, Hq, d = q.shape
    outs = []
    for t in (o_hist, o_curr):
        outs.append(torch.empty_like(q) if t is None else t)
    lses = []
    for t in (lse_hist, lse_curr):
        lses.append(torch.empty((B, Hq, q_len), dtype=torch.float32, device=q.device)
                    if t is None else t)
    _check("bsx_bsa_prefill_split", lib.bsx_bsa_prefill_split(
        shape_of(q, k), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), q_len, q_start_pos,
        _ptr(outs[0]), _ptr(lses[0]), _ptr(outs[1]), _ptr(lses[1]), _stream(stream)))
    return outs[0], lses[0], outs[1], lses[1]


def bsx_chunk_prefill(q, k, v, q_start_pos: int, stride: int, threshold: float, *,
                      mask=None, o=None, lse=None, workspace=None, stream=None):
    """Estimate + block-sparse attention over all key blocks -> (mask, o, lse)."""
    lib = load()
    B, q_len, Hq, _ = q.shape
    Lk = k.shape[1]
    shape = shape_of(q, k)
    if mask is None:
        mask = torch.empty((B, Hq, q_len // 128, Lk // 128), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, q_len), dtype=torch.float32, device=q.device)
    need = lib.bsx_chunk_prefill_workspace_bytes(shape, q_len, q_start_pos, stride)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check("bsx_chunk_prefill", lib.bsx_chunk_prefill(
        shape, _ptr(q), _ptr(k), _ptr(v), q_len, q_start_pos, stride, float(threshold),
        _ptr(mask), _ptr(o), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return mask, o, lse


def bsx_chunk_step(q, k, v, q_start_pos: int, stride: int, threshold: float, *,
                   cpu_block_tokens: int = 1024, mask=None, o=None, lse=None, o_curr=None,
                   lse_curr=None, keep=None, with_keep: bool = True, workspace=None,
                   stream=None):
    """The chunk step (estimate, attention on history and current chunk, LSE
    merge, CPU-block flags) -> (mask, o, lse, keep); keep is None when there
    is no history CPU block or with_keep is False.  o_curr / lse_curr are
    scratch."""
    lib = load()
    B, q_len, Hq, _ = q.shape
    Lk = k.shape[1]
    shape = shape_of(q, k)
    dev = q.device
    if mask is None:
        mask = torch.empty((B, Hq, q_len // 128, Lk // 128), dtype=torch.uint8, device=dev)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, q_len), dtype=torch.float32, device=dev)
    if o_curr is None:
        o_curr = torch.empty_like(q)
    if lse_curr is None:
        lse_curr = torch.empty((B, Hq, q_len), dtype=torch.float32, device=dev)
    n_cpu = q_start_pos // cpu_block_tokens
    if keep is None and with_keep and n_cpu > 0:
        keep = torch.empty((B, n_cpu), dtype=torch.uint8, device=dev)
    need = lib.bsx_chunk_prefill_workspace_bytes(shape, q_len, q_start_pos, stride)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check("bsx_chunk_step", lib.bsx_chunk_step(
        shape, _ptr(q), _ptr(k), _ptr(v), q_len, q_start_pos, stride, float(threshold),
        cpu_block_tokens, _ptr(mask), _ptr(o), _ptr(lse), _ptr(o_curr), _ptr(lse_curr),
        _ptr(keep), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return mask, o, lse, keep


def bsx_merge_attn(o1, lse1, o2, lse2, *, stream=None):
    """In-place LSE merge of (o2, lse2) into (o1, lse1); returns (o1, lse1)."""
    lib = load()
    B, q_len, Hq, d = o1.shape
    shape = BsxShape(B, Hq, Hq, d, _dtype_code(o1))
    _check("bsx_merge_attn", lib.bsx_merge_attn(
        shape, q_len, _ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _stream(stream)))
    return o1, lse1


def bsx_map_mask_to_cpu_blocks(mask, q_start_pos: int, cpu_block_tokens: int = 1024,
                               force_first_last: bool = False, *, keep=None, stream=None):
    """uint8 keep flags [B, q_start_pos / cpu_block_tokens] from a block mask."""
    lib = load()
    B, Hq, nqb, nkb = mask.shape
    n_cpu = q_start_pos // cpu_block_tokens
    if keep is None:
        keep = torch.empty((B, max(n_cpu, 0)), dtype=torch.uint8, device=mask.device)
    shape = BsxShape(B, Hq, Hq, 128, BSX_BF16)
    flags = BSX_FORCE_FIRST_LAST if force_first_last else 0
    _check("bsx_map_mask_to_cpu_blocks", lib.bsx_map_mask_to_cpu_blocks(
        shape, _ptr(mask), nqb * 128, q_start_pos, cpu_block_tokens, flags,
        _ptr(keep) if keep.numel() else None, _stream(stream)))
    return keep


def bsx_cpu_block_mask(keep, q_len: int, q_start_pos: int, Hq: int,
                       cpu_block_tokens: int = 1024, *, mask=None, stream=None):
    """Offload-mode BSA block mask [B, Hq, q_len/128, Lk/128] from keep flags."""
    lib = load()
    B = keep.shape[0]
    nkb = (q_start_pos + q_len) // 128
    if mask is None:
        mask = torch.empty((B, Hq, q_len // 128, nkb), dtype=torch.uint8, device=keep.device)
    shape = BsxShape(B, Hq, Hq, 128, BSX_BF16)
    _check("bsx_cpu_block_mask", lib.bsx_cpu_block_mask(
        shape, _ptr(keep) if keep.numel() else None, q_len, q_start_pos, cpu_block_tokens,
        _ptr(mask), _stream(stream)))
    return mask


def bsx_debug_drop_ring_item(cta: int, item: int) -> None:
    """Failure-path test hook: the calling thread's next bf16 attention launch
    has CTA `cta` stop loading before K/V ring item `item`, so its bounded
    waits run out and the error word records it (see bsxattn.h)."""
    _check("bsx_debug_drop_ring_item", load().bsx_debug_drop_ring_item(cta, item))


def bsx_debug_fused_skip_row(row: int) -> None:
    """Failure-path test hook: the calling thread's next fused chunk step never
    marks selection row `row` ready, so that row's attention CTA's bounded
    wait runs out and the error word records it (see bsxattn.h)."""
    _check("bsx_debug_fused_skip_row", load().bsx_debug_fused_skip_row(row))


def bsx_chunk_prefill_workspace_bytes(shape: BsxShape, q_len: int, q_start_pos: int,
                                      stride: int) -> int:
    """Device workspace bytes of bsx_chunk_prefill (0 for invalid arguments)."""
    return int(load().bsx_chunk_prefill_workspace_bytes(shape, q_len, q_start_pos, stride))


def bsx_last_error(stream=None) -> int:
    """Wait for `stream` (default: torch's current stream), read and clear the
    device error word; returns the raw word (0 = none)."""
    lib = load()
    status = lib.bsx_last_error(_stream(stream))
    if status not in (0, -4):
        raise BsxError("bsx_last_error", status)
    return int(lib.bsx_last_error_code())


def make_chunk_buffers(q_host, k_host, q_start_pos: int, stride: int,
                       cpu_block_tokens: int = 1024, *, offload: bool = False,
                       e4m3_estimate: bool = False, fused: bool = False,
                       with_keep: bool = True, device=None) -> dict:
    """Device buffers for bsx_chunk_step_host, allocated once by the caller
    (torch) and reused across steps; the library allocates nothing."""
    device = torch.device("cuda") if device is None else torch.device(device)
    B, q_len, Hq, d = q_host.shape
    Lk, Hkv = k_host.shape[1], k_host.shape[2]
    dt = q_host.dtype
    u8 = torch.uint8
    n_cpu = q_start_pos // cpu_block_tokens
    shape = BsxShape(B, Hq, Hkv, d, _dtype_code(q_host))
    # the step may run as one fused kernel: room for its control block
    need = max(load().bsx_estimate_workspace_bytes(shape, q_len, q_start_pos, stride),
               load().bsx_chunk_prefill_workspace_bytes(shape, q_len, q_start_pos, stride))
    mshape = (B, Hq, q_len // 128, Lk // 128)
    return {
        "q": torch.empty(q_host.shape, dtype=dt, device=device),
        "k": torch.empty(k_host.shape, dtype=dt, device=device),
        "v": torch.empty(k_host.shape, dtype=dt, device=device),
        "mask": torch.empty(mshape, dtype=u8, device=device),
        "bsa_mask": torch.empty(mshape, dtype=u8, device=device) if offload else None,
        "o": torch.empty(q_host.shape, dtype=dt, device=device),
        "lse": torch.empty((B, Hq, q_len), dtype=torch.float32, device=device),
        "o_curr": None if fused else torch.empty(q_host.shape, dtype=dt, device=device),
        "lse_curr": None if fused else torch.empty((B, Hq, q_len), dtype=torch.float32,
                                                   device=device),
        "keep": (torch.empty((B, n_cpu), dtype=u8, device=device)
                 if n_cpu > 0 and (with_keep or offload) else None),
        "q8": torch.empty(q_host.shape, dtype=u8, device=device) if e4m3_estimate else None,
        "k8": torch.empty(k_host.shape, dtype=u8, device=device) if e4m3_estimate else None,
        "workspace": torch.empty(max(int(need), 16), dtype=u8, device=device),
        "done": _recorded_event(device),
    }


def _recorded_event(device):
    """A CUDA event that exists (torch creates events on first record)."""
    ev = torch.cuda.Event()
    ev.record(torch.cuda.current_stream(device))
    return ev


def bsx_chunk_step_host(q_host, k_host, v_host, q_start_pos: int, stride: int,
                        threshold: float, *, buffers: dict, o_host=None, lse_host=None,
                        keep_host=None, cpu_block_tokens: int = 1024,
                        force_first_last: bool = False, offload: bool = False,
                        e4m3_estimate: bool = False, fused: bool = False, stream=None,
                        upload_stream=None, download_stream=None):
    """The chunk step from (pinned) host q/k/v to host (o, lse, keep); the
    results are valid once `download_stream` (default: `stream`) has
    completed, or buffers["done"] has (see bsxattn.h)."""
    lib = load()
    B, q_len, Hq, d = q_host.shape
    Hkv = k_host.shape[2]
    n_cpu = q_start_pos // cpu_block_tokens
    if o_host is None:
        o_host = torch.empty(q_host.shape, dtype=q_host.dtype, pin_memory=True)
    if lse_host is None:
        lse_host = torch.empty((B, Hq, q_len), dtype=torch.float32, pin_memory=True)
    with_keep = n_cpu > 0 and buffers.get("keep") is not None
    if keep_host is None and with_keep:
        keep_host = torch.empty((B, n_cpu), dtype=torch.uint8, pin_memory=True)
    done = buffers.get("done")
    bufs = BsxChunkBuffers(*[None if buffers.get(n) is None else _ptr(buffers[n]).value
                             for n in
                             ("q", "k", "v", "mask", "bsa_mask", "o", "lse", "o_curr",
                              "lse_curr", "keep", "q8", "k8", "workspace")],
                           buffers["workspace"].numel(),
                           None if done is None else done.cuda_event)
    flags = ((BSX_FORCE_FIRST_LAST if force_first_last else 0) |
             (BSX_STEP_OFFLOAD if offload else 0) |
             (BSX_STEP_E4M3_ESTIMATE if e4m3_estimate else 0) |
             (BSX_STEP_FUSED if fused else 0))
    us = None if upload_stream is None else ctypes.c_void_p(upload_stream.cuda_stream)
    ds = None if download_stream is None else ctypes.c_void_p(download_stream.cuda_stream)
    _check("bsx_chunk_step_host", lib.bsx_chunk_step_host(
        BsxShape(B, Hq, Hkv, d, _dtype_code(q_host)), _hptr(q_host), _hptr(k_host),
        _hptr(v_host), q_len, q_start_pos, stride, float(threshold), cpu_block_tokens, flags,
        ctypes.byref(bufs), _hptr(o_host), _hptr(lse_host),
        _hptr(keep_host) if with_keep else None, _stream(stream), us, ds))
    return o_host, lse_host, keep_host
