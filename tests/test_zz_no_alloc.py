"""aq_gemv_nvfp4_noalloc: the GEMV for callers that cannot allocate device
memory.  Its split-K scratch is a fixed array inside the library, so the
call takes no workspace; its output must equal aq_gemv_nvfp4 on the same
(register-decode) kernel with a caller workspace bit for bit, call after
call, and so also stay within the GEMV tolerance of that output.

The file name makes pytest collect it last, so it runs both after every
other test in the session and, run on its own, as the first library call
in a fresh process (where the call also sets the scratch up)."""
import numpy as np
import pytest
import torch

from gpu_helpers import DEV, assert_gemv_close, gemv_gpu, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def as_ref(y):
    return y.float().cpu().numpy().astype(np.float64)


def test_noalloc_matches_workspace_gemv_on_consecutive_calls():
    # 1B-shaped fused gate+up at m = 1, then 31B-shaped down at m = 3: two
    # calls in a row on one stream, sharing the one scratch array
    cases = [((13824, 1152), 1, 31), ((5376, 21504), 3, 32)]
    ws_, xs, refs, outs = [], [], [], []
    for (n, k), m, seed in cases:
        assert aq.gemv_workspace_bytes(n, k, m) <= aq.NOALLOC_MAX_SCRATCH
        w = quantize_gpu(inputs.weight(n, k, seed=seed, device=DEV))
        x = inputs.tokens(m, k, seed=seed + 100, device=DEV)
        ws_.append(w)
        xs.append(x)
        # the existing entry point, own workspace, on the kernel this entry
        # point runs (the register-decode kernel)
        refs.append(gemv_gpu(w, x, path=aq.PATH_GEMV_REGDECODE))
        outs.append(torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    for rep in range(2):
        for w, x, y in zip(ws_, xs, outs):
            y.fill_(float("nan"))
            aq.gemv_noalloc(w, x, y)
        torch.cuda.synchronize()
        assert aq.poll_device_status() == aq.OK
        for i, (y, ref) in enumerate(zip(outs, refs)):
            # the header promises the workspace call's bits; the tolerance
            # check is a second, looser statement of the same
            assert torch.equal(y, ref), "round %d case %d: outputs differ" % (rep, i)
            assert_gemv_close(y, as_ref(ref), "round %d case %d" % (rep, i))


def test_noalloc_rejects_paths_it_does_not_run():
    # m = 17 on AQ_PATH_AUTO would take the MMA path in aq_gemv_nvfp4, and
    # AQ_PATH_MMA always does; this entry point runs the register-decode
    # kernel only, so both are refused on the host before any launch
    n, k = 256, 512
    w = quantize_gpu(inputs.weight(n, k, seed=5, device=DEV))
    for m, path in ((17, aq.PATH_AUTO), (4, aq.PATH_MMA), (2, aq.PATH_GEMV_TCGEN05)):
        x = inputs.tokens(m, k, seed=6, device=DEV)
        y = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(aq.AqError) as exc:
            aq.gemv_noalloc(w, x, y, path=path)
        assert exc.value.status == aq.ERR_UNSUPPORTED, (m, path)
        assert "register-decode" in str(exc.value)
        assert not y.any()
    assert aq.poll_device_status() == aq.OK


def test_noalloc_rejects_a_weight_beyond_the_scratch():
    # [2^19, 1024]: thousands of row blocks, far more partial sums than the
    # fixed scratch holds.  The buffers are real and full-sized, so the call
    # is rejected on the host with nothing out of bounds even in principle.
    n, k = 1 << 19, 1024
    need = aq.gemv_workspace_bytes(n, k, 1)
    if need <= aq.NOALLOC_MAX_SCRATCH:
        pytest.skip("this device's split needs only %d bytes" % need)
    w = aq.Nvfp4Weight(n, k, torch.zeros(aq.packed_bytes(n, k), dtype=torch.uint8, device=DEV),
                       torch.zeros(aq.scale_bytes(n, k), dtype=torch.uint8, device=DEV),
                       torch.ones(1, dtype=torch.float32, device=DEV))
    x = torch.zeros((1, k), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((1, n), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(aq.AqError) as exc:
        aq.gemv_noalloc(w, x, y)
    assert exc.value.status == aq.ERR_WORKSPACE
    assert "static scratch" in str(exc.value)
    assert aq.poll_device_status() == aq.OK
