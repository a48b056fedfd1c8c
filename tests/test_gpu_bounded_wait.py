"""Failure detection on the GPU without a fault: every barrier wait in the library's kernels
is bounded by GPU time and, once the limit passes, raises TQ_FLAG_TIMEOUT and lets the kernel
return.  tq_check_bounded_wait runs that same wait on a barrier nothing arrives at; the host
then reads TQ_ERR_TIMEOUT, the flag is cleared by the read, and the context stays usable."""
import pytest
import torch

from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300 import api

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports_timeout():
    B.load()
    B.tq_device_status()                      # start from a clear status word
    stream = torch.cuda.current_stream().cuda_stream
    assert B.tq_check_bounded_wait(1000, stream) == B.TQ_OK   # 1 ms limit
    st, flags = B.tq_device_status()
    assert st == B.TQ_ERR_TIMEOUT and flags & B.TQ_FLAG_TIMEOUT, (st, flags)
    assert B.tq_device_status() == (B.TQ_OK, 0)
    # the context is still usable: a quantise call right after runs and reports nothing
    x = torch.randn(1, 1, 64, 128, device="cuda").to(torch.bfloat16)
    kc = api.Codec.prod(3)
    cache = api.ProdCache.empty(1, 1, 64, 3)
    api.quantize_prod(kc, x, cache)
    assert B.tq_device_status() == (B.TQ_OK, 0)
    torch.testing.assert_close(cache.xnorm[0, 0], x[0, 0].float().norm(dim=-1), rtol=1e-5, atol=0)
