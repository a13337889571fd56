"""The benchmark's algorithmic work per step, against the closed forms of the workloads
(32 sequences x 32768 positions, K = 2048, 128 heads)."""
import bench
import dsa_inputs as di


def test_decode_32k_bytes_and_flops():
    wl = di.preset("decode_32k")
    w = bench.algorithmic(wl, 32 * 2048)
    assert w["k_bytes"] == 32 * 32768 * 128 * 2 == 268_435_456
    assert w["gather_bytes"] == 32 * 2048 * 576 * 2 == 75_497_472
    assert w["metric_bytes"] == 343_932_928
    assert w["li_flop"] == 32 * 32768 * 64 * 128 * 2
    assert w["sfa_flop"] == 32 * 2048 * 128 * (576 + 512) * 2


def test_quantised_indexer_and_latent_cache_bytes():
    # e4m3 keys: 128 B per row plus a 4-byte scale (per-token FP8) or four E8M0 bytes (MXFP8)
    for name in ("decode_32k_fp8", "decode_32k_mxfp8"):
        assert bench.algorithmic(di.preset(name), 32 * 2048)["k_bytes"] == 138_412_032
    # FP8 latent rows of 608 bytes
    assert bench.algorithmic(di.preset("decode_32k_kv8"), 32 * 2048)["gather_bytes"] == 32 * 2048 * 608


def test_prefill_indexer_flops_follow_the_causal_triangle():
    wl = di.preset("prefill_64k")
    w = bench.algorithmic(wl, 0)
    visible = sum(61440 + i + 1 for i in range(4096))
    assert w["li_flop"] == visible * 64 * 128 * 2
