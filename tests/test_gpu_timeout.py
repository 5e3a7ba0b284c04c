"""Device-side waits are bounded: an injected missing arrival makes one block's
waits run out, the kernel stops cleanly, the status word reports it, and the
CUDA context stays usable.  No memory fault, trap or unbounded wait is used:
the injection only skips one copy and its barrier arrival."""

import pytest
import torch

from tests.conftest import cuda_available
from tests.parity import compare, oracle_out, run_gpu, seeded

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


def test_wait_budget_runs_out_cleanly(lib):
    from chunked_prefill_attention_gb300 import q8attn as Q
    q = seeded((1, 128, 1, 64), 1, "cuda", torch.float16)
    k = seeded((1, 128, 1, 64), 2, "cuda")
    v = seeded((1, 128, 1, 64), 3, "cuda")
    k8 = Q.q8kv_quantize(k)
    v8 = Q.q8kv_quantize(v)
    st = Q.State(1, 1, 128, "cuda")
    rc, _ = Q.device_status(clear=True)
    assert rc == Q.Q8A_OK
    assert Q.status() == Q.Q8A_OK
    Q.set_wait_timeout_ns(50_000_000)
    try:
        Q.test_inject(1)
        Q.attn_chunk_step(q, k8, v8, 0, 128, st)
        torch.cuda.current_stream().synchronize()
        # the sync-free check sees the failure through the host-mapped word
        assert Q.status(torch.cuda.current_stream()) == Q.Q8A_ERR_TIMEOUT
        rc, status = Q.device_status(clear=True)
        assert rc == Q.Q8A_ERR_TIMEOUT
        assert status & 1 and ((status >> 8) & 0xFF) in (1, 2, 3, 4, 5)
        assert Q.status() == Q.Q8A_OK   # cleared with the device word
    finally:
        Q.test_inject(0)
        Q.set_wait_timeout_ns(2_000_000_000)
    # the context is still usable and results are right afterwards
    out, *_ = run_gpu(q, k, v, 128)
    rc, status = Q.device_status(clear=True)
    assert rc == Q.Q8A_OK and status == 0
    assert Q.status() == Q.Q8A_OK
    want, *_ = oracle_out(q, k, v)
    compare(out.cpu().numpy(), want, "after timeout")
