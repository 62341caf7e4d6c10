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
