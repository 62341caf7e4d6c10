"""The bench's byte accounting (CPU): the weight bytes of the two decode-step
workloads follow from 0.5625 B per element (AttnQuant docs, "Throughput",
"What quantization actually saves"), and the algorithmic bytes a step must
move add the fp32 tensor scale, the bf16 activations read and the bf16
outputs written per projection."""
import bench
from nvfp4_block_scaled_aq_gb300 import inputs


def test_weight_bytes_are_0_5625_per_element():
    for shapes, layers, total in ((inputs.LAYER_31B, inputs.LAYERS_31B, 13_934_592_000),
                                  (inputs.LAYER_1B, inputs.LAYERS_1B, 392_491_008)):
        elements = sum(n * k for n, k in shapes) * layers
        assert bench.weight_bytes(shapes, layers) == total == elements * 9 // 16


def test_algorithmic_bytes_add_scale_activations_and_outputs():
    for m in (1, 4):
        extra = sum(4 + 2 * m * k + 2 * m * n for n, k in inputs.LAYER_31B) * inputs.LAYERS_31B
        got = bench.algorithmic_bytes(inputs.LAYER_31B, inputs.LAYERS_31B, m)
        assert got == bench.weight_bytes(inputs.LAYER_31B, inputs.LAYERS_31B) + extra
    assert bench.algorithmic_bytes(inputs.LAYER_31B, inputs.LAYERS_31B, 1) == 13_946_389_440


def test_load_time_bytes_are_2_5625_per_element_plus_the_bundle():
    """A load-time call reads the bf16 weight once (2 B per element) and
    writes 0.5 B of nibbles and 1/16 B of E4M3 scales per element plus the
    4-byte g_dec: 41/16 B per element.  The fused form also reads s (fp32
    per row) and the rank-r U and V (bf16).  The totals are the ones the
    load-time leg reports for its three shapes."""
    for n, k in ((43008, 5376), (13824, 1152), (1152, 6912)):
        plain = bench.load_time_bytes(n, k, 4, False)
        assert plain == n * k * 41 // 16 + 4
        assert bench.load_time_bytes(n, k, 4, True) - plain == 4 * n + 2 * (n + k) * 4
    assert bench.load_time_bytes(43008, 5376, 4, False) == 592_478_212
    assert bench.load_time_bytes(43008, 5376, 4, True) == 593_037_316
    assert bench.load_time_bytes(13824, 1152, 4, True) == 40_983_556
    assert bench.load_time_bytes(1152, 6912, 4, True) == 20_473_348
