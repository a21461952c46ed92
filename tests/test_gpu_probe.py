"""The block-scaled MMA rate probe runs on the GPU and returns a plausible dense rate
(the kind::mxf8f6f4 MMAs of the expert GEMMs run at the FP8 tensor rate: nominal 4.5
PFLOP/s dense on a GB300; the check only bounds it loosely)."""
import pytest

from moe_testlib import build_lib

pytestmark = pytest.mark.gpu


def test_mma_rate_probe():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    m = build_lib()
    for n in (16, 64, 192):
        tf, ms = m.moe_probe_mma_rate(0, 20000, n)
        assert 10.0 < tf < 20000.0, (n, tf)
        assert ms > 0.0
