"""The allocation-free estimate entry point, called through the C ABI.

bsx_xattn_estimate_noalloc serves callers that may not allocate device memory
and have no buffer to lend as scratch (for instance a plugin whose host engine
owns all device memory): it uses a fixed 32 MiB scratch array held in the
library's device code.  Its results must equal those of bsx_xattn_estimate
with a caller workspace, call after call, since every call reuses (and must
fully rewrite) the same scratch.  This file sorts last so that a run stopping
at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from block_sparse_long_xattn_gb300 import _lib as L
from block_sparse_long_xattn_gb300 import bsx_xattn_estimate
from block_sparse_long_xattn_gb300.inputs import make_workload
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # two calls in a row with different problems: a second call must not see
    # anything the first one left in the shared scratch
    dict(seed=41, B=1, Hq=8, Hkv=2, d=128, Lk=4096, q_start_pos=3072, alpha=3.0, n_hot=4,
         dtype="bf16", stride=8, tau=0.95),
    dict(seed=42, B=2, Hq=4, Hkv=1, d=64, Lk=2048, q_start_pos=1024, alpha=2.0, n_hot=2,
         dtype="f32", stride=16, tau=0.9),
]


def _noalloc(lib, q, k, P, S, tau, mask, A):
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bsx_xattn_estimate_noalloc(
        L.shape_of(q, k), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        q.shape[1], P, S, tau, ctypes.c_void_p(mask.data_ptr()),
        ctypes.c_void_p(A.data_ptr()), st)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    lib = L.load()
    for c in CASES:
        c = dict(c)
        S, tau = c.pop("stride"), c.pop("tau")
        w = make_workload(**c)
        q, k = to_dev(w.q, w.dtype), to_dev(w.k, w.dtype)
        B, Lq, Hq, _ = q.shape
        shape = (B, Hq, Lq // 128, k.shape[1] // 128)
        A_ref = torch.zeros(shape, dtype=torch.float32, device="cuda")
        m_ref = bsx_xattn_estimate(q, k, w.q_start_pos, S, tau, block_sums=A_ref)
        A = torch.full(shape, -1.0, dtype=torch.float32, device="cuda")
        m = torch.full(shape, 7, dtype=torch.uint8, device="cuda")
        assert _noalloc(lib, q, k, w.q_start_pos, S, tau, m, A) == 0
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical results
        assert torch.equal(m, m_ref)
        assert torch.equal(A, A_ref)
        assert L.bsx_last_error() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = L.load()
    # 32 q-heads, 1024 key blocks, 512 reshaped rows -> 64 MiB > 32 MiB
    s = L.BsxShape(1, 32, 8, 128, L.BSX_BF16)
    p = ctypes.c_void_p(256)
    assert lib.bsx_xattn_estimate_noalloc(s, p, p, 4096, 126976, 8, 0.9, p, None, None) == -5
    # an invalid stride is reported as the regular entry point reports it
    assert lib.bsx_xattn_estimate_noalloc(s, p, p, 4096, 0, 3, 0.9, p, None, None) == -2
