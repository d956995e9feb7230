"""dsa_topk_noalloc against dsa_topk, through the C ABI.

dsa_topk_noalloc serves callers that may not allocate device memory (a
plugin given only a stream, a real-time thread that must not take allocator
locks, a process whose device memory is divided up in advance): its scratch
is one fixed array inside the library, reused by every call.  These tests
check that it selects exactly what dsa_topk selects with a caller-owned
workspace, and what the CPU oracle selects, on consecutive calls of different shapes (so that what one call
leaves in the array cannot leak into the next), and that a problem too big
for the array is refused before anything runs.

The file name sorts last on purpose: a run that stops at the first failure
has run every other test before this one.  It must pass on its own in a
fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_common import lib, need_gpu

pytestmark = pytest.mark.gpu


def _scores(seed, Nq, ld, n_lo):
    """Integer scores in [0, 5) (heavy ties, decided by position), one row of
    normals, and eligible counts in [n_lo, ld]."""
    rng = np.random.default_rng(seed)
    s = rng.integers(0, 5, size=(Nq, ld)).astype(np.float32)
    s[0] = rng.standard_normal(ld).astype(np.float32)
    n = rng.integers(n_lo, ld + 1, size=Nq).astype(np.int32)
    return torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()


def _with_workspace(dsa, scores, n, K):
    Nq, ld = scores.shape
    idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    rc = dsa.lib().dsa_topk(ctypes.c_void_p(scores.data_ptr()), ld, ctypes.c_void_p(n.data_ptr()),
                            Nq, K, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                            ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dsa.lib().dsa_last_error_string()
    return idx


def _no_alloc(dsa, scores, n, K):
    Nq, ld = scores.shape
    idx = torch.full((Nq, K), 7, dtype=torch.int32, device="cuda")
    rc = dsa.lib().dsa_topk_noalloc(ctypes.c_void_p(scores.data_ptr()), ld,
                                    ctypes.c_void_p(n.data_ptr()), Nq, K,
                                    ctypes.c_void_p(idx.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dsa.lib().dsa_last_error_string()
    return idx


def test_no_alloc_topk_matches_dsa_topk_on_consecutive_calls():
    need_gpu()
    dsa = lib()
    # 1: rows of 120000 positions (three blocks: the array holds block winners)
    # 2: a different, single-block problem right after it
    # 3: the first problem again, over what call 2 left in the array
    problems = ((1, 6, 120000, 2048, 60000), (2, 33, 20000, 512, 1), (1, 6, 120000, 2048, 60000))
    for seed, Nq, ld, K, n_lo in problems:
        assert dsa.topk_workspace_size(Nq, ld, K) <= dsa.TOPK_NOALLOC_SCRATCH_BYTES
        scores, n = _scores(seed, Nq, ld, n_lo)
        want = _with_workspace(dsa, scores, n, K)
        got = _no_alloc(dsa, scores, n, K)
        torch.cuda.synchronize()
        assert torch.equal(got, want), (seed, Nq, ld, K)
        # and both are the oracle's selection (full sort by score desc,
        # position asc; ascending output, -1 padding)
        ref = oracle.topk(scores.cpu().numpy(), n.cpu().numpy(), K)
        np.testing.assert_array_equal(got.cpu().numpy(), ref, err_msg=str((seed, Nq, ld, K)))


def test_no_alloc_topk_refuses_a_problem_beyond_its_scratch():
    need_gpu()
    dsa = lib()
    Nq, ld, K = 64, 100000, 16384    # three blocks per row, 16384 winners each
    assert dsa.topk_workspace_size(Nq, ld, K) > dsa.TOPK_NOALLOC_SCRATCH_BYTES
    scores = torch.zeros((Nq, ld), dtype=torch.float32, device="cuda")
    n = torch.full((Nq,), ld, dtype=torch.int32, device="cuda")
    idx = torch.full((Nq, K), 7, dtype=torch.int32, device="cuda")
    before = dsa.launch_count()
    rc = dsa.lib().dsa_topk_noalloc(ctypes.c_void_p(scores.data_ptr()), ld,
                                    ctypes.c_void_p(n.data_ptr()), Nq, K,
                                    ctypes.c_void_p(idx.data_ptr()), None)
    assert rc == -3                                   # DSA_ERR_WORKSPACE
    assert b"scratch" in dsa.lib().dsa_last_error_string()
    assert dsa.launch_count() == before               # nothing launched
    torch.cuda.synchronize()
    assert bool((idx == 7).all())                     # output untouched
