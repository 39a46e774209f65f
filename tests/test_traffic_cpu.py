"""The algorithmic byte model (the roofline numerator) against the per-layer-
step totals worked out for the scope table before any kernel: StreamingLLM
1.077 GB, H2O MHA 0.273 GB, H2O GQA 0.548 GB, Random 1.351 GB plus its
position-table read, H2O on the Random shape 1.364 GB; and the score-storage
variants differing by exactly their per-slot score bytes."""
import pytest

from workloads import configs, traffic


@pytest.mark.parametrize("name,gb,digits", [("sink_window", 1.077, 3), ("h2o_mha", 0.273, 3),
                                            ("h2o_gqa", 0.548, 3), ("h2o_reasoning", 1.364, 3)])
def test_totals_match_the_scope_table(name, gb, digits):
    w = configs.get(name)
    assert round(traffic.steady_layer_step_bytes(w) / 1e9, digits) == gb


def test_random_total_is_the_kv_total_plus_the_position_table():
    """The scope table's Random total (1.351 GB) counts the attended K/V and
    the small per-token terms; the model also counts the 4-byte position
    table read every step (4 * C per unit), which the table's per-unit
    formula lists."""
    w = configs.get("random")
    units = w.batch * w.n_kv_heads
    got = traffic.steady_layer_step_bytes(w)
    assert abs((got - units * 4 * w.capacity) / 1e9 - 1.351) < 0.0005


def test_sink_window_from_first_principles():
    w = configs.get("sink_window")  # B=64, 32 KV heads, C=1024, d=128, bf16, G=1
    per_unit = (1024 + 1) * 2 * 128 * 2 + 2 * 128 * 2 + 2 * 1 * 128 * 2
    assert traffic.steady_layer_step_bytes(w) == 64 * 32 * per_unit


def test_score_storage_variants_differ_by_their_score_bytes():
    fp32, half, int8 = (traffic.steady_layer_step_bytes(configs.get(n))
                        for n in ("h2o_mha", "h2o_fp16scores", "h2o_int8scores"))
    units, C = 16 * 32, 1024
    assert fp32 - half == units * (4 * C + 2)
    assert fp32 - int8 == units * (6 * C - 1)


def test_kv_cache_size_formula_matches_the_pages_sizing():
    """2 (K and V) x 80 layers x 8 KV heads x 128 x 2 bytes x 32K tokens =
    10.74 GB, the pages' figure for a 70B-class GQA model."""
    assert round(traffic.kv_cache_bytes(80, 8, 128, 2, 32768) / 1e9, 2) == 10.74
