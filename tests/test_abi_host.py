"""Host-side checks of the C ABI (no GPU needed).

The shared library must load, export every entry point include/bsxattn.h
declares, and reject bad arguments on the host before touching the device.
None of these calls launches a kernel.
"""
import ctypes
import os
import re

import pytest

from block_sparse_long_xattn_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsxattn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsx_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from block_sparse_long_xattn_gb300 import build
        build.build()
    return L.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert names, "no entry points parsed from the header"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in bsxattn.h but not exported"
    assert set(L.EXPORTS) <= set(names)


def test_version_and_status_strings(lib):
    assert lib.bsx_version() >= 1
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert lib.bsx_status_string(code)


def test_workspace_formula(lib):
    s = L.BsxShape(1, 32, 8, 128, L.BSX_BF16)
    # one float per (b, q-head, key block, reshaped row)
    assert lib.bsx_estimate_workspace_bytes(s, 4096, 28672, 8) == 32 * 256 * 512 * 4
    assert lib.bsx_estimate_workspace_bytes(s, 4096, 126976, 16) == 32 * 1024 * 256 * 4
    assert lib.bsx_estimate_workspace_bytes(s, 4000, 0, 8) == 0      # q_len not /128
    assert lib.bsx_estimate_workspace_bytes(s, 4096, 0, 3) == 0      # bad stride


def test_chunk_prefill_workspace_formula(lib):
    s = L.BsxShape(1, 32, 8, 128, L.BSX_BF16)
    # the partials (rounded up to 256 bytes), then the fused launch's control
    # block: 4 counters, tiles_done per (b, h, 128-row tile of reshaped rows),
    # then per (b, h, q-block) the row's ready flag, 4 bytes each, rounded up
    # to 256; then one
    # float per (b, h, 256-key tile of the last row tile, reshaped row),
    # rounded up to 256
    est = 32 * 256 * 512 * 4
    ctl = (4 + 32 * (512 // 128 + 4096 // 128)) * 4
    n_kt = (28672 // 8 + 512 - 1) // 256 + 1            # 16 key tiles at 32K
    assert lib.bsx_chunk_prefill_workspace_bytes(s, 4096, 28672, 8) == \
        est + (ctl + 255) // 256 * 256 + 32 * n_kt * 512 * 4
    tiny = L.BsxShape(1, 1, 1, 64, L.BSX_BF16)
    assert lib.bsx_estimate_workspace_bytes(tiny, 128, 0, 16) == 32
    assert lib.bsx_chunk_prefill_workspace_bytes(tiny, 128, 0, 16) == 256 + 256 + 256
    assert lib.bsx_chunk_prefill_workspace_bytes(s, 4000, 0, 8) == 0   # q_len not /128
    assert lib.bsx_chunk_prefill_workspace_bytes(s, 4096, 0, 3) == 0   # bad stride


def test_chunk_prefill_rejects_bad_arguments(lib):
    s = L.BsxShape(1, 4, 2, 128, L.BSX_BF16)
    p = ctypes.c_void_p(64)
    need = lib.bsx_chunk_prefill_workspace_bytes(s, 512, 1024, 8)

    def call(shape=s, stride=8, tau=0.9, v=p, ws=need, wp=p):
        return lib.bsx_chunk_prefill(shape, p, p, v, 512, 1024, stride, tau, p, p, p, wp, ws,
                                     None)
    assert call(stride=3) == -2
    assert call(tau=float("nan")) == -1
    assert call(tau=0.0) == -1
    assert call(v=None) == -1
    assert call(v=ctypes.c_void_p(72)) == -1                        # misaligned
    assert call(shape=L.BsxShape(1, 3, 2, 128, 1)) == -1            # Hq % Hkv
    assert call(ws=need - 1) == -5                                  # no room for the control block
    assert call(wp=None) == -5


def test_chunk_step_rejects_bad_arguments(lib):
    s = L.BsxShape(1, 4, 2, 128, L.BSX_BF16)
    p = ctypes.c_void_p(64)
    need = lib.bsx_chunk_prefill_workspace_bytes(s, 512, 1024, 8)

    def call(stride=8, tau=0.9, cpu=256, o_curr=p, keep=p, ws=need):
        return lib.bsx_chunk_step(s, p, p, p, 512, 1024, stride, tau, cpu, p, p, p, o_curr, p,
                                  keep, p, ws, None)
    assert call(stride=3) == -2
    assert call(tau=float("nan")) == -1
    assert call(o_curr=None) == -1                  # the current chunk's scratch is required
    assert call(o_curr=ctypes.c_void_p(72)) == -1   # misaligned
    assert call(cpu=100) == -1                      # CPU blocks: multiples of 128
    assert call(cpu=768) == -1                      # ... dividing q_start_pos
    assert call(ws=need - 1) == -5
    assert call(cpu=100, keep=None, ws=need - 1) == -5  # without keep the block size is unused


def test_debug_fused_skip_row_hook(lib):
    assert lib.bsx_debug_fused_skip_row(3) == 0          # arm ...
    assert lib.bsx_debug_fused_skip_row(-1) == 0         # ... and disarm (no launch here)


NULL = None


def _est(lib, shape, q_len=1024, P=0, stride=8, tau=0.9, ptr=16, ws=1 << 30):
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.bsx_xattn_estimate(shape, p, p, q_len, P, stride, tau, p, None, p, ws, None)


def test_estimate_rejects_bad_arguments(lib):
    good = L.BsxShape(1, 4, 2, 128, L.BSX_BF16)
    assert _est(lib, L.BsxShape(1, 3, 2, 128, 1)) == -1          # Hq % Hkv
    assert _est(lib, L.BsxShape(1, 4, 2, 96, 1)) == -2           # head dim
    assert _est(lib, L.BsxShape(1, 4, 2, 128, 5)) == -2          # dtype
    assert _est(lib, good, q_len=1000) == -1                     # q_len % 128
    assert _est(lib, good, P=100) == -1                          # q_start_pos % 128
    assert _est(lib, good, stride=3) == -2                       # stride
    assert _est(lib, good, tau=0.0) == -1                        # threshold
    assert _est(lib, good, tau=float("nan")) == -1
    assert _est(lib, good, ptr=0) == -1                          # null pointers
    assert _est(lib, good, ptr=8) == -1                          # misaligned
    assert _est(lib, good, ws=16) == -5                          # workspace too small


def test_bsa_merge_map_reject_bad_arguments(lib):
    s = L.BsxShape(1, 4, 2, 128, L.BSX_BF16)
    p = ctypes.c_void_p(16)
    # kb range outside [0, Lk/128]
    assert lib.bsx_bsa_prefill(s, p, p, p, p, 256, 256, 2, 1, p, p, None) == -1
    assert lib.bsx_bsa_prefill(s, p, p, p, p, 256, 256, 0, 5, p, p, None) == -1
    assert lib.bsx_bsa_prefill(s, p, None, p, p, 256, 256, 0, 4, p, p, None) == -1
    # split launch: every output required, q_start_pos a multiple of 128
    assert lib.bsx_bsa_prefill_split(s, p, p, p, p, 256, 256, p, p, None, p, None) == -1
    assert lib.bsx_bsa_prefill_split(s, p, p, p, p, 256, 200, p, p, p, p, None) == -1
    assert lib.bsx_merge_attn(s, 100, p, p, p, p, None) == -1
    assert lib.bsx_merge_attn(s, 128, p, None, p, p, None) == -1
    # cpu block size must divide q_start_pos and be a multiple of 128
    assert lib.bsx_map_mask_to_cpu_blocks(s, p, 128, 4096, 1000, 0, p, None) == -1
    assert lib.bsx_map_mask_to_cpu_blocks(s, p, 128, 4096, 3072, 0, p, None) == -1
    assert lib.bsx_map_mask_to_cpu_blocks(s, p, 128, 4096, 1024, 4, p, None) == -1


def test_mask_size_limit(lib):
    """Calls that use the block mask index it with 32-bit grids: a mask of more
    than 2^31 - 1 elements is unsupported, rejected before any launch; the
    merge, which has no mask, takes the same rows."""
    p = ctypes.c_void_p(16)
    big = L.BsxShape(1024, 32, 8, 128, L.BSX_BF16)   # 1024*32*32*2048 = 2^31 mask elements
    assert lib.bsx_bsa_prefill(big, p, p, p, p, 4096, 258048, 0, 1, p, p, None) == -2
    assert lib.bsx_bsa_prefill_split(big, p, p, p, p, 4096, 258048, p, p, p, p, None) == -2
    assert lib.bsx_map_mask_to_cpu_blocks(big, p, 4096, 258048, 1024, 0, p, None) == -2
    assert lib.bsx_estimate_workspace_bytes(big, 4096, 258048, 8) == 0
    ok = L.BsxShape(1023, 32, 8, 128, L.BSX_BF16)    # one batch fewer fits
    assert lib.bsx_bsa_prefill(ok, p, p, p, p, 4096, 258048, 0, 1, p, None, None) == -1
    # the merge sees no mask: only its own arguments are checked
    assert lib.bsx_merge_attn(big, 4096, p, None, p, p, None) == -1


def _host_step(lib, shape=None, q_len=256, P=1024, stride=8, tau=0.9, cpu=1024, flags=0,
               host=64, ws=1 << 30, drop=(), **set_fields):
    """bsx_chunk_step_host with fake, aligned, never-dereferenced pointers:
    every case below must be rejected before anything is enqueued."""
    shape = shape or L.BsxShape(1, 4, 2, 128, L.BSX_BF16)
    fields = {n: 4096 for n in ("q", "k", "v", "mask", "bsa_mask", "o", "lse", "o_curr",
                                "lse_curr", "keep", "q8", "k8", "workspace")}
    fields.update(set_fields)
    for n in drop:
        fields[n] = None
    bufs = L.BsxChunkBuffers(*[fields[n] for n in (
        "q", "k", "v", "mask", "bsa_mask", "o", "lse", "o_curr", "lse_curr", "keep", "q8", "k8",
        "workspace")], ws, None)
    h = ctypes.c_void_p(host) if host else None
    return lib.bsx_chunk_step_host(shape, h, h, h, q_len, P, stride, tau, cpu, flags,
                                   ctypes.byref(bufs), h, h, h, None, None, None)


def test_chunk_step_host_rejects_bad_arguments(lib):
    assert _host_step(lib, host=0) == -1                              # host inputs required
    assert lib.bsx_chunk_step_host(L.BsxShape(1, 4, 2, 128, 1), ctypes.c_void_p(64),
                                   ctypes.c_void_p(64), ctypes.c_void_p(64), 256, 1024, 8, 0.9,
                                   1024, 0, None, ctypes.c_void_p(64), ctypes.c_void_p(64),
                                   None, None, None, None) == -1    # no device buffers
    assert _host_step(lib, shape=L.BsxShape(1, 4, 2, 128, L.BSX_F8E4M3)) == -2  # e4m3 in
    assert _host_step(lib, shape=L.BsxShape(1, 3, 2, 128, 1)) == -1   # Hq % Hkv
    assert _host_step(lib, stride=3) == -2
    assert _host_step(lib, tau=float("nan")) == -1
    assert _host_step(lib, q_len=200) == -1
    assert _host_step(lib, cpu=1000) == -1                            # cpu block % 128
    assert _host_step(lib, P=1536, cpu=1024) == -1                    # cpu block divides P
    assert _host_step(lib, o=4100) == -1                              # misaligned output
    assert _host_step(lib, drop=("keep",)) == -1                      # keep_host needs keep
    assert _host_step(lib, cpu=0) == -1                               # no division by zero
    assert _host_step(lib, flags=2, drop=("keep",)) == -1             # offload needs keep
    assert _host_step(lib, flags=16) == -1                            # unknown flag
    assert _host_step(lib, drop=("o_curr",)) == -1                    # split needs o_curr
    assert _host_step(lib, flags=2, drop=("bsa_mask",)) == -1         # offload needs its mask
    assert _host_step(lib, flags=4, drop=("k8",)) == -1               # e4m3 needs its copies
    assert _host_step(lib, flags=4, shape=L.BsxShape(1, 4, 2, 64, 1)) == -2  # e4m3: d = 128
    assert _host_step(lib, ws=16) == -5                               # workspace too small
    est_only = lib.bsx_estimate_workspace_bytes(L.BsxShape(1, 4, 2, 128, 1), 256, 1024, 8)
    assert _host_step(lib, flags=8, ws=est_only) == -5                # fused: + control block


def test_debug_drop_hook_arguments(lib):
    assert lib.bsx_debug_drop_ring_item(0, -1) == -1     # armed needs an item
    assert lib.bsx_debug_drop_ring_item(0, 3) == 0       # arm ...
    assert lib.bsx_debug_drop_ring_item(-1, 0) == 0      # ... and disarm (no launch here)


def test_binding_requires_cuda_tensors():
    import torch
    q = torch.zeros(1, 128, 2, 64)
    with pytest.raises((ValueError, RuntimeError)):
        L.bsx_bsa_prefill(q, q[:, :, :1], q[:, :, :1], torch.ones(1, 2, 1, 1, dtype=torch.uint8), 0)
