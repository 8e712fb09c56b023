"""The benchmark's workload description: byte counts from the shapes, and the
one config dict both arms print (host only)."""
import bench
import workloads as wl


def test_cycle_weight_bytes_from_first_principles():
    # 4-bit nibbles plus one bf16 scale and one bf16 bias per 64 weights:
    # 0.5 + 4/64 bytes per weight, over 64 layers of seven projections and
    # the LM head
    per_layer = 4 * 5120 * 5120 + 2 * 17408 * 5120 + 17408 * 5120
    weights = 64 * per_layer + 151936 * 5120
    assert bench.cycle_bytes_static(3)[0] == weights // 2 + weights // 64 * 4
    assert bench.cycle_bytes_static(3)[0] == 13838376960


def test_cycle_algorithmic_bytes_grow_with_depth():
    w3, a3 = bench.cycle_bytes_static(3)
    w5, a5 = bench.cycle_bytes_static(5)
    assert w3 == w5 and a5 > a3 > w3
    # M = K + 1 bf16 rows in and fp32 rows out per projection, and the
    # GatedDeltaNet tape work, are what the depth adds
    shapes = [(N, K) for _ in range(wl.N_LAYERS) for _, N, K in wl.LAYER_PROJECTIONS]
    shapes.append((wl.VOCAB, wl.HIDDEN))
    rows = sum(2 * K + 4 * N for N, K in shapes)
    T3, T5, H, d = 4, 6, wl.GDN_HEADS, wl.GDN_DIM
    # q, k, v, alpha, beta in; outputs; tape records (e, k, alpha) per head
    per_token = H * (3 * d + 2) * 4 + H * d * 4 + 4 * H * (2 * d + 1)
    assert a5 - a3 == 2 * rows + wl.N_LAYERS * (T5 - T3) * per_token


def test_both_arms_print_the_same_config():
    c = bench.cycle_config(3)
    assert c == bench.cycle_config(3, "plans", 1)
    assert {"workload", "depth_K", "M", "batch", "weight_bytes_per_cycle",
            "algorithmic_bytes_per_cycle"} <= set(c)
    assert c["M"] == 4 and c["batch"] == 1
