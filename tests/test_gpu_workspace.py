"""One workspace shared by every GEMV path, shape and token count in turn:
each call must leave the workspace as the next call needs it (tickets and
the zero region back at zero), so every result equals the same call made
with a fresh zero-filled workspace, bit for bit."""
import pytest
import torch

from gpu_helpers import DEV, gemv_gpu, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def test_shared_workspace_across_paths_shapes_and_token_counts():
    shapes = [(8192, 5376), (5376, 21504), (1536, 1152)]
    ws_ = {s: quantize_gpu(inputs.weight(*s, seed=900 + i, device=DEV)) for i, s in enumerate(shapes)}
    # (shape, m, path): split row blocks through the zero region (m <= 8) and
    # through the ticket-counted partials (m > 8), with the tcgen05 and MMA
    # paths writing their own partials and buffers in between
    calls = [
        (shapes[0], 1, aq.PATH_GEMV_REGDECODE), (shapes[1], 3, aq.PATH_GEMV_REGDECODE),
        (shapes[0], 24, aq.PATH_MMA), (shapes[0], 1, aq.PATH_GEMV_REGDECODE),
        (shapes[2], 2, aq.PATH_GEMV_TCGEN05), (shapes[1], 12, aq.PATH_GEMV_REGDECODE),
        (shapes[1], 3, aq.PATH_GEMV_REGDECODE), (shapes[2], 64, aq.PATH_MMA),
        (shapes[2], 8, aq.PATH_GEMV_REGDECODE), (shapes[0], 16, aq.PATH_GEMV_REGDECODE),
        (shapes[0], 1, aq.PATH_GEMV_REGDECODE),
    ]
    size = max(aq.gemv_workspace_bytes(n, k, m) for (n, k), m, _ in calls)
    shared = torch.zeros(size, dtype=torch.uint8, device=DEV)
    for i, ((n, k), m, path) in enumerate(calls):
        x = inputs.tokens(m, k, seed=950 + i, device=DEV)
        y_shared = gemv_gpu(ws_[(n, k)], x, ws=shared, path=path)
        y_fresh = gemv_gpu(ws_[(n, k)], x, path=path)
        torch.cuda.synchronize()
        assert torch.equal(y_shared, y_fresh), "call %d: [%d, %d] m=%d path %d" % (i, n, k, m, path)
        assert aq.poll_device_status() == aq.OK
    # after the sequence the first region of the workspace is back at zero
    assert not shared[: 12 << 20].any()
