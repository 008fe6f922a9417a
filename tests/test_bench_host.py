"""Host-side arithmetic of bench.py (CPU): the interval union behind the in-step kernel-class
times, and the algorithmic byte counts the rooflines divide by."""
import bench
from synth.recipes import MISTRAL_7B


def test_interval_union():
    assert bench.interval_union_ns([]) == 0
    assert bench.interval_union_ns([(0, 10)]) == 10
    assert bench.interval_union_ns([(0, 10), (5, 12), (20, 25)]) == 17   # overlap, then a gap
    assert bench.interval_union_ns([(20, 25), (0, 10), (10, 11)]) == 16  # unsorted, touching
    assert bench.interval_union_ns([(0, 100), (10, 20), (30, 40)]) == 100  # nested


def test_byte_counts():
    s = MISTRAL_7B
    w = s.weight_bytes_per_step()
    assert w == 2 * 7_110_393_856
    # projections: weights plus the fp32 activations in and out, about 2 MB a layer at B = 8
    extra = bench.projection_bytes(s, 8) - w
    assert 32 * 1.5e6 < extra < 32 * 2.5e6
    # attention: 131072 bytes of KV per live position per row, plus the appended one
    assert bench.attention_bytes(s, [99], 16) > 101 * 131072
    assert abs(bench.attention_bytes(s, [9999], 8) / bench.attention_bytes(s, [9999], 16) - 1.0625 / 2) < 0.01
