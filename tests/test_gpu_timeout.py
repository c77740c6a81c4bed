"""The bounded-wait path on the GPU, without faulting anything: a test kernel
waits on an mbarrier nothing arrives at, gives up after a short limit and
records a timeout; the host sees ATTN_ERR_TIMEOUT, attention launched while
the record stands skips its work, and clearing the record restores normal
operation (the CUDA context stays usable throughout)."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_recorded_reported_and_cleared(cuda_dev):
    import sequence_attn_fwd_gb300 as sa

    sa.query_device_error()  # start clean
    st = torch.cuda.current_stream().cuda_stream
    assert sa.lib.attn_debug_expire_wait(20_000, st) == 0  # 20 ms
    with pytest.raises(sa.AttnError) as ei:
        sa.query_device_error()
    assert ei.value.status == 4  # ATTN_ERR_TIMEOUT
    sa.query_device_error()  # the record was cleared by the first query


def test_recorded_timeout_makes_later_launches_skip_until_cleared(cuda_dev):
    import sequence_attn_fwd_gb300 as sa

    w = workloads.Workload("adhoc", 1, 2, 2, 384, 128, True, 1, 99)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    o_ok, lse_ok = sa.attn_fwd(q, k, v, causal=True)
    o_ok, lse_ok = o_ok.clone(), lse_ok.clone()
    st = torch.cuda.current_stream().cuda_stream
    assert sa.lib.attn_debug_expire_wait(10_000, st) == 0
    o_skip, lse_skip = sa.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert (o_skip == 0).all() and torch.isneginf(lse_skip).all()
    with pytest.raises(sa.AttnError):
        sa.query_device_error()
    o2, lse2 = sa.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, o_ok) and torch.equal(lse2, lse_ok)
    sa.query_device_error()
