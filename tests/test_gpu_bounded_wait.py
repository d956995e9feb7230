"""The give-up path of the bounded waits, exercised without a hang: a wait on
an mbarrier that nothing completes must end after its limit with
DSA_STATUS_TIMEOUT in the workspace status, and the context must stay usable
(a full pipeline runs correctly right after)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import DevicePipeline, lib, need_gpu

pytestmark = pytest.mark.gpu

DSA_STATUS_TIMEOUT = 0x8


def _selftest(dsa, expire, limit_ns, ws):
    rc = dsa.lib().dsa_selftest_bounded_wait(int(expire), ctypes.c_uint64(limit_ns),
                                             ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, dsa.lib().dsa_last_error_string()


def test_wait_that_nothing_completes_gives_up_and_reports():
    need_gpu()
    dsa = lib()
    ws = dsa.workspace(256)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    _selftest(dsa, True, 20_000_000, ws)            # 20 ms limit
    ev1.record()
    torch.cuda.synchronize()
    assert ev0.elapsed_time(ev1) >= 19.0           # it waited for its limit ...
    assert dsa.get_status(ws) == DSA_STATUS_TIMEOUT  # ... then reported instead of hanging
    _selftest(dsa, False, 20_000_000, ws)           # completed barrier: no report
    torch.cuda.synchronize()
    assert dsa.get_status(ws) == 0
    # the context is still usable: a small pipeline matches the oracle
    c = W.make_case("after-timeout", seed=900, seq_lens=(300, 129), K=64, Hq=16, Dqk=128, Dv=128,
                    latent=False, H_i=4, D_i=64, idx_dtype="bf16")
    g = DevicePipeline(c, dsa=dsa)
    g.all()
    s_ref = oracle.index_score(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq, c.q_pos,
                               c.q_idx, c.w, c.kidx_pool, oracle.BF16, c.max_len)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy(), oracle.topk(s_ref, c.n_elig, c.K))
    assert g.status() == 0


def test_selftest_rejects_limits_outside_its_range():
    need_gpu()
    dsa = lib()
    ws = dsa.workspace(256)
    n0 = dsa.launch_count()
    for bad in (0, 10, 2_000_000_000):
        rc = dsa.lib().dsa_selftest_bounded_wait(1, ctypes.c_uint64(bad), ctypes.c_void_p(ws.data_ptr()),
                                                 ws.numel(), None)
        assert rc == -1
    assert dsa.launch_count() == n0
