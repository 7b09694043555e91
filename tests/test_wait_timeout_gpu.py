"""The bounded-wait path on the GPU without a fault: a kernel whose only
mbarrier wait is never satisfied gives up after 20 ms, records its site in the
device error word and returns; the host reads the code, the word is cleared by
the read, and the context stays usable for a correct attention call."""
import pytest
import torch

from oracle import reference as ref
from paged_attention_relative_gb300.workloads import make_case
from tests.gpu_util import assert_close, run

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_reports_its_site_and_returns():
    import paged_attention_relative_gb300 as pa
    assert pa.device_error() == 0
    pa.check_wait_timeout(20)
    assert pa.device_error() == pa.SITE_SELF_TEST
    assert pa.device_error() == 0          # reading clears it
    c = make_case(seed=31, seqlens_q=[1, 70], seqlens_k=[300, 200], num_heads=8, num_kv_heads=2,
                  head_dim=128, rel_extent=32)
    assert_close(run(c), ref.forward(c), what="after a timed-out wait")
    assert pa.device_error() == 0
