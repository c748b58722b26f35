"""bench.py's accounting, pinned by hand arithmetic (CPU only): the algorithmic
bytes and flops the roofline divides by, and the kernels per forward it
reports as gpu_launches."""
import numpy as np

import bench
import workloads as W


def _counts(E, touched):
    c = np.zeros(E, np.int64)
    c[:touched] = 1
    return c


def test_fp4_small_decode_bytes_by_hand():
    wl = W.WORKLOADS["small_decode"]          # T=8, H=2048, I=512, E=256, k=8
    a = bench.algorithmic(wl, _counts(256, 56))
    # per expert W1: 2I rows x (H/2 packed E2M1 + H/32 UE8M0) = 1024 x 1088 B
    w1 = 1024 * (1024 + 64)
    x_q = 8 * (2048 + 64)                      # FP8 tokens + UE8M0 per 32
    h_q = 64 * (512 + 16)                      # FP8 h + UE8M0 per 32, per pair
    assert a["gemm1_bytes"] == 56 * w1 + x_q + h_q == 62440960
    # per expert W2: H rows x (I/2 + I/32) = 2048 x 272 B; pair rows in BF16
    assert a["gemm2_bytes"] == 56 * 2048 * 272 + h_q + 64 * 2048 * 2
    assert a["gemm1_flops"] == 2 * 64 * 1024 * 2048
    assert a["layer_flops"] == 2 * 64 * 3 * 2048 * 512
    assert a["layer_bytes"] == 8 * 2048 * 2 + 8 * 256 * 4 + 56 * (w1 + 2048 * 272) + 8 * 2048 * 2


def test_bfp8_small_decode_bytes_by_hand():
    wl = W.WORKLOADS["small_decode"]
    a = bench.algorithmic_bfp8(wl, _counts(256, 56))
    # per expert W1: 1024 x 2048 E4M3 + (1024/128) x (2048/128) float32 block scales
    w1 = 1024 * 2048 + 8 * 16 * 4
    x_q = 8 * (2048 + 16 * 4)                  # FP8 tokens + a float32 per 128
    h_q = 64 * (512 + 4 * 4)
    assert a["gemm1_bytes"] == 56 * w1 + x_q + h_q == 117519872
    # W2: 2048 x 512 + 16 x 4 scales; FP32 weighted pair rows
    assert a["gemm2_bytes"] == 56 * (2048 * 512 + 16 * 4 * 4) + h_q + 64 * 2048 * 4
    assert a["touched_experts"] == 56


def test_launches_per_forward():
    # small problems: front kernel + one launch of GEMM1 + GEMM2 + combine
    assert bench.launches_per_forward(8, 2048, 512, 256, 8) == 2
    assert bench.launches_per_forward_bfp8(8, 2048, 256, 8) == 2
    # large decode (16-token tiles): route, permute (one launch for <= 2048 pairs), pool cast, GEMM1, GEMM2, combine
    assert bench.launches_per_forward(128, 7168, 2048, 256, 8) == 6
    assert bench.launches_per_forward_bfp8(128, 7168, 256, 8) == 6
    # prefill (CTA pairs, default schedule): route, permute (count + scatter), token-order cast, GEMM1, GEMM2, combine
    assert bench.launches_per_forward(4096, 7168, 2048, 256, 8) == 7
    # ... under the expert-wave schedule: GEMM1 + GEMM2 + combine in one launch
    assert bench.launches_per_forward(4096, 7168, 2048, 256, 8, schedule=2) == 5
    assert bench.single_gemm_launch(4096, 7168, 2048, 256, 8, schedule=2)
    assert not bench.single_gemm_launch(4096, 7168, 2048, 256, 8)
    assert bench.single_gemm_launch(8, 2048, 512, 256, 8)
    assert not bench.single_gemm_launch(128, 7168, 2048, 256, 8, schedule=2)
    # H/128 odd: one-CTA 224-token tiles, separate GEMM launches
    assert not bench.pair_tiles(4096, 7168 - 128, 2048, 256, 8)
    assert not bench.single_gemm_launch(4096, 7168 - 128, 2048, 256, 8, schedule=2)


def test_layer_rates():
    alg = {"layer_bytes": 94_000_000, "layer_flops": 402_653_184}
    r = bench.layer_rates(alg, 0.0394)                 # 39.4 us per step
    assert r["gbs"] == round(94e6 / 39.4e-6 / 1e9, 1)
    assert r["tflops"] == round(402653184 / 39.4e-6 / 1e12, 3)


def test_traffic_table_lookup():
    # every kernel family names existing sources and a SHA-256; a workload or
    # launch without a capture reads as "not captured", a captured one gives
    # bytes (while its sources still hash to the recorded value) or says why not
    for fam in bench.TRAFFIC.values():
        assert len(fam["src_sha256"]) == 64
        assert bench.gemm_sources_sha256(fam["sources"])
    assert bench.measured_traffic("tiny", "fused", 1000) == (None, "not captured")
    assert bench.measured_traffic("large_decode", "gemm1", 1000) == (None, "not captured")
    fresh = bench.gemm_sources_sha256(bench.PAIR_SOURCES) == bench.TRAFFIC["pair"]["src_sha256"]
    nbytes, how = bench.measured_traffic("prefill", "gemm1", 10**9)
    if fresh:
        ratio = bench.TRAFFIC["pair"]["prefill"]["gemm1"]["ratio"]
        assert nbytes == round(ratio * 10**9) and "prefill_e32" in how
    else:
        assert nbytes is None and "changed" in how
