"""GPU tests of the per-step weight stream: one launch per (fused)
projection, in stream order, with and without programmatic dependent
launch, and replayed from a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemv_close, bits, gemv_gpu, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def build_stack(layers, shapes, m, seed=0):
    ws, Ws, xs, ys = [], [], [], []
    for layer in range(layers):
        for p, (n, k) in enumerate(shapes):
            W = inputs.weight(n, k, seed=inputs.seed_of(seed, layer, p), device=DEV)
            Ws.append(W)
            ws.append(quantize_gpu(W))
            xs.append(inputs.tokens(m, k, seed=inputs.seed_of(seed + 1, layer, p), device=DEV))
            ys.append(torch.empty((m, n), dtype=torch.bfloat16, device=DEV))
    return Ws, ws, xs, ys


def step_workspace(shapes, m):
    size = max(aq.gemv_workspace_bytes(n, k, m) for n, k in shapes)
    return torch.zeros(size, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("m", [1, 4])
@pytest.mark.parametrize("flags", [0, aq.STEP_PDL])
def test_step_equals_separate_gemvs(m, flags):
    Ws, ws, xs, ys = build_stack(3, inputs.LAYER_1B, m)
    wsp = step_workspace(inputs.LAYER_1B, m)
    args = aq.StepArgs(ws, xs, ys)
    aq.decode_step(args, wsp, flags=flags)
    torch.cuda.synchronize()
    for w, x, y in zip(ws, xs, ys):
        assert torch.equal(y, gemv_gpu(w, x))
    assert aq.poll_device_status() == aq.OK


def test_step_graph_replay_matches_eager():
    m = 1
    Ws, ws, xs, ys = build_stack(2, inputs.LAYER_1B, m, seed=3)
    wsp = step_workspace(inputs.LAYER_1B, m)
    args = aq.StepArgs(ws, xs, ys)
    aq.decode_step(args, wsp)
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        aq.decode_step(args, wsp, stream=side)  # warm-up outside capture
        side.synchronize()
        for y in ys:
            y.zero_()
        with torch.cuda.graph(graph, stream=side):
            aq.decode_step(args, wsp, stream=side)
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(ys, eager):
        assert torch.equal(a, b)


def test_full_1b_step_against_oracle():
    """All 26 layers x 4 projections of the 1B-shaped stack in one step;
    one seeded projection per kind checked against the oracle in full."""
    m = 1
    Ws, ws, xs, ys = build_stack(inputs.LAYERS_1B, inputs.LAYER_1B, m, seed=7)
    wsp = step_workspace(inputs.LAYER_1B, m)
    aq.decode_step(aq.StepArgs(ws, xs, ys), wsp)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    for p in range(4):
        i = int(rng.integers(inputs.LAYERS_1B)) * 4 + p
        packed, scales, ge, gd = oracle.quantize(bits(Ws[i]))
        y_ref = oracle.gemv(packed, scales, gd, bits(xs[i]))
        assert_gemv_close(ys[i], y_ref, "projection %d" % i)


# ------------------------------------------------------------ persistent step

@pytest.mark.parametrize("m", [1, 3, 12])
def test_persistent_step_matches_oracle_and_separate_calls(m):
    """One cooperative launch for the whole stack: every projection within
    tolerance of the oracle, and equal bit for bit to the per-projection
    launch on the register-decode kernel (same partition, same form)."""
    Ws, ws, xs, ys = build_stack(3, inputs.LAYER_1B, m, seed=11)
    plan = aq.StepPlan(ws, xs, ys)
    wsp = plan.workspace()
    aq.step_run(plan, wsp)
    torch.cuda.synchronize()
    assert aq.poll_device_status() == aq.OK
    for i, (W, w, x, y) in enumerate(zip(Ws, ws, xs, ys)):
        packed, scales, ge, gd = oracle.quantize(bits(W))
        y_ref = oracle.gemv(packed, scales, gd, bits(x))
        assert_gemv_close(y, y_ref, "projection %d" % i)
        assert torch.equal(y, gemv_gpu(w, x, path=aq.PATH_GEMV_REGDECODE)), "projection %d" % i
    # the counters are back at zero: a second run on the same workspace
    # gives the same bits
    first = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    aq.step_run(plan, wsp)
    torch.cuda.synchronize()
    assert aq.poll_device_status() == aq.OK
    for a, b in zip(ys, first):
        assert torch.equal(a, b)


def test_persistent_step_repeats_bit_exact_and_is_m_invariant():
    Ws, ws, xs4, ys4 = build_stack(2, inputs.LAYER_31B[:2], 4, seed=12)
    plan4 = aq.StepPlan(ws, xs4, ys4)
    wsp = plan4.workspace()
    aq.step_run(plan4, wsp)
    torch.cuda.synchronize()
    first = [y.clone() for y in ys4]
    aq.step_run(plan4, wsp)
    torch.cuda.synchronize()
    for a, b in zip(ys4, first):
        assert torch.equal(a, b)
    # two of the four tokens alone: the same bits
    xs2 = [x[2:4].contiguous() for x in xs4]
    ys2 = [torch.empty((2, y.shape[1]), dtype=torch.bfloat16, device=DEV) for y in ys4]
    plan2 = aq.StepPlan(ws, xs2, ys2)
    aq.step_run(plan2, plan2.workspace())
    torch.cuda.synchronize()
    for a, b in zip(ys2, first):
        assert torch.equal(a, b[2:4])
    # one token takes the one-token kernel form: held to the oracle
    xs1 = [x[2:3].contiguous() for x in xs4]
    ys1 = [torch.empty((1, y.shape[1]), dtype=torch.bfloat16, device=DEV) for y in ys4]
    plan1 = aq.StepPlan(ws, xs1, ys1)
    aq.step_run(plan1, plan1.workspace())
    torch.cuda.synchronize()
    for i, (W, x, a) in enumerate(zip(Ws, xs1, ys1)):
        packed, scales, ge, gd = oracle.quantize(bits(W))
        assert_gemv_close(a, oracle.gemv(packed, scales, gd, bits(x)), "one token, projection %d" % i)
    assert aq.poll_device_status() == aq.OK


def test_persistent_step_in_a_cuda_graph():
    Ws, ws, xs, ys = build_stack(2, inputs.LAYER_1B, 1, seed=13)
    plan = aq.StepPlan(ws, xs, ys)
    wsp = plan.workspace()
    aq.step_run(plan, wsp)
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for y in ys:
            y.zero_()
        with torch.cuda.graph(graph, stream=side):
            aq.step_run(plan, wsp, stream=side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(ys, eager):
        assert torch.equal(a, b)


def test_persistent_step_rejects_mismatched_run_on_device():
    """A run whose m or workspace does not match its plan launches, finds
    the mismatch on the device before touching memory, and reports it."""
    Ws, ws, xs, ys = build_stack(1, inputs.LAYER_1B, 1, seed=14)
    plan = aq.StepPlan(ws, xs, ys)
    wsp = plan.workspace()
    aq.step_run(plan, wsp, m=2)
    assert aq.poll_device_status() == aq.ERR_INVALID_ARG
    small = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    aq.step_run(plan, small)
    assert aq.poll_device_status() == aq.ERR_INVALID_ARG
    aq.step_run(plan, wsp)
    assert aq.poll_device_status() == aq.OK


@pytest.mark.parametrize("flag", ["regdecode", "tcgen05", "mma"])
def test_step_kernel_flags_match_their_single_calls(flag):
    """aq_decode_step_weights with a kernel flag gives, projection by
    projection, exactly the single call on that kernel's path."""
    m = 2
    Ws, ws, xs, ys = build_stack(2, inputs.LAYER_1B, m, seed=15)
    fl = {"regdecode": aq.STEP_REGDECODE, "tcgen05": aq.STEP_TCGEN05, "mma": aq.STEP_MMA}[flag]
    path = {"regdecode": aq.PATH_GEMV_REGDECODE, "tcgen05": aq.PATH_GEMV_TCGEN05,
            "mma": aq.PATH_MMA}[flag]
    size = max(aq.gemv_workspace_bytes(n, k, m) for n, k in inputs.LAYER_1B)
    wsp = torch.zeros(size, dtype=torch.uint8, device=DEV)
    aq.decode_step(aq.StepArgs(ws, xs, ys), wsp, flags=aq.STEP_PDL | fl)
    torch.cuda.synchronize()
    for w, x, y in zip(ws, xs, ys):
        assert torch.equal(y, gemv_gpu(w, x, path=path))
    assert aq.poll_device_status() == aq.OK


def test_step_rejects_two_kernel_flags():
    Ws, ws, xs, ys = build_stack(1, inputs.LAYER_1B[:1], 1, seed=16)
    wsp = step_workspace(inputs.LAYER_1B[:1], 1)
    with pytest.raises(aq.AqError) as e:
        aq.decode_step(aq.StepArgs(ws, xs, ys), wsp, flags=aq.STEP_REGDECODE | aq.STEP_MMA)
    assert e.value.status == aq.ERR_INVALID_ARG


# ------------------------------------------------------------ full size, bench path

def _sampled_31b_check(Ws_bits, ws, xs, ys, layers, what):
    rng = np.random.default_rng(31)
    for i in range(layers * 4):
        n, k = inputs.LAYER_31B[i % 4]
        Wb = Ws_bits[i]
        ge, gd = oracle.global_scales(oracle.amax(Wb))
        rows = np.sort(rng.choice(n, 256, replace=False))
        packed_r, scales_r = oracle.quantize_rows(Wb[rows], ge)
        y_ref = oracle.gemv(packed_r, scales_r, gd, bits(xs[i]))
        assert_gemv_close(ys[i][:, rows], y_ref, "%s, projection %d" % (what, i))


def test_31b_step_pdl_graph_sampled_parity():
    """Two layers of the ~31B-shaped stack at full size through the timed
    path of the benchmark: aq_decode_step_weights with programmatic
    dependent launch and the next-projection L2 prefetch, captured in a CUDA
    graph and replayed; 256 seeded rows of every projection against the
    oracle."""
    layers, m = 2, 1
    Ws_bits, ws, xs, ys = [], [], [], []
    for layer in range(layers):
        for p, (n, k) in enumerate(inputs.LAYER_31B):
            W = inputs.weight(n, k, seed=inputs.seed_of(0, layer, p), device=DEV)
            ws.append(quantize_gpu(W))
            Ws_bits.append(bits(W))
            del W
            xs.append(inputs.tokens(m, k, seed=inputs.seed_of(1, layer, p), device=DEV))
            ys.append(torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV))
    wsp = step_workspace(inputs.LAYER_31B, m)
    args = aq.StepArgs(ws, xs, ys)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        aq.decode_step(args, wsp, flags=aq.STEP_PDL | aq.STEP_REGDECODE, stream=side)
        side.synchronize()
        for y in ys:
            y.fill_(float("nan"))
        with torch.cuda.graph(graph, stream=side):
            aq.decode_step(args, wsp, flags=aq.STEP_PDL | aq.STEP_REGDECODE, stream=side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert aq.poll_device_status() == aq.OK
    _sampled_31b_check(Ws_bits, ws, xs, ys, layers, "PDL graph")
    # the persistent step on the same stack: the same bits
    chain = [y.clone() for y in ys]
    plan = aq.StepPlan(ws, xs, ys)
    aq.step_run(plan, plan.workspace())
    torch.cuda.synchronize()
    assert aq.poll_device_status() == aq.OK
    for i, (a, b) in enumerate(zip(ys, chain)):
        assert torch.equal(a, b), "persistent step differs from the chain at projection %d" % i


@pytest.mark.parametrize("flag", ["regdecode", "mma"])
@pytest.mark.parametrize("m", [1, 4])
def test_step_chained_projections_wait_for_their_inputs(flag, m):
    """Each projection's input is the previous projection's output (square
    weights, x of projection p + 1 aliasing y of projection p), launched as
    one step with programmatic dependent launch: every kernel that reads x
    (the GEMV's activation staging, the MMA path's activation quantisation)
    must wait for the kernel that wrote it.  The result equals the same
    chain run call by call."""
    n = 1152
    layers = [(n, n)] * 6
    ws = [quantize_gpu(inputs.weight(n, n, seed=inputs.seed_of(31, 0, p), device=DEV))
          for p in range(len(layers))]
    x0 = inputs.tokens(m, n, seed=32, device=DEV)
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for _ in layers]
    xs = [x0] + ys[:-1]
    fl = {"regdecode": aq.STEP_REGDECODE, "mma": aq.STEP_MMA}[flag]
    path = {"regdecode": aq.PATH_GEMV_REGDECODE, "mma": aq.PATH_MMA}[flag]
    wsp = step_workspace(layers, m)
    aq.decode_step(aq.StepArgs(ws, xs, ys), wsp, flags=aq.STEP_PDL | fl)
    torch.cuda.synchronize()
    x = x0
    for i, w in enumerate(ws):
        y = gemv_gpu(w, x, path=path)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], y), "projection %d" % i
        x = y
    assert aq.poll_device_status() == aq.OK
