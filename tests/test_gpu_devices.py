"""Device placement in the Python binding.

Each call runs on the GPU that holds its first tensor, and on that GPU's current
stream. Tensors spread over several devices are rejected before any launch."""
import pytest

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_calls_reject_tensors_on_another_device():
    from exact_attention_flash_gb300 import fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(1, 1, 64, 64, 5, "cuda", with_do=False)
    with pytest.raises(ValueError):
        fa_forward(q, k.cpu(), v)
    with pytest.raises(ValueError):
        fa_forward(q.cpu(), k, v)
