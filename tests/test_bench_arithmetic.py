"""The benchmark's roofline arithmetic (CPU): the algorithmic bytes and FLOPs it divides by are
the counts the workloads' definitions give, written out here term by term."""
import bench
from workloads import DECODE_CONFIG, scan_config, ssd_config


def test_scan_compulsory_bytes_of_the_layer_workloads():
    # (batch, dim, seqlen), N = 16, bf16 in and out: u, delta, z read and y written (2 B each),
    # B and C read, A (dim x 16 fp32), D and delta_bias (dim fp32), final state written.
    for name, (b, d, L) in {"c1_mamba130m": (8, 1536, 2048), "c2_mamba2p8b": (4, 5120, 2048),
                            "c3_long_1m": (1, 1536, 1 << 20)}.items():
        want = b * d * L * 8 + 2 * b * 16 * L * 2 + d * 16 * 4 + 2 * d * 4 + b * d * 16 * 4
        assert bench.scan_algorithmic_bytes(scan_config(name)) == want, name
    assert bench.scan_algorithmic_bytes(scan_config("c2_mamba2p8b")) == 337_747_968


def test_scan_compulsory_bytes_fp32_tiny_workload():
    # C0 (1, 64, 256) fp32: 4 B per activation element in and out.
    want = 64 * 256 * 16 + 2 * 16 * 256 * 4 + 64 * 16 * 4 + 2 * 64 * 4 + 64 * 16 * 4
    assert bench.scan_algorithmic_bytes(scan_config("c0_tiny_f32")) == want


def test_decode_bytes_per_layer_step():
    # state read and written (fp32), x, dt, z read and out written (bf16), B and C (bf16),
    # A (fp32), D and dt_bias (fp32).
    d = DECODE_CONFIG.dim
    for batch, want in ((1, 1_065_024), (16, 11_510_784), (64, 44_937_216)):
        assert bench.decode_algorithmic_bytes(batch, d, 16) == want
    # with the short convolution: its bf16 window of 4 read and written, fp32 taps and bias
    extra = 64 * d * 4 * 2 * 2 + d * 4 * 4 + d * 4
    assert bench.decode_algorithmic_bytes(64, d, 16, conv=True) == 44_937_216 + extra


def test_ssd_flops_and_bytes_of_the_mamba2_layer():
    cfg = ssd_config("ssd1_mamba2_2p7b")
    alg, executed, byts = bench.ssd_work(cfg)
    Q, N, P = 128, 128, 64
    chunks = 4 * 80 * (2048 // Q)
    per_chunk = 2 * Q * Q * N + 2 * Q * Q * P + 2 * Q * N * P + 2 * Q * N * P  # C B^T, M X, C S, B^T (wX)
    assert alg == chunks * per_chunk
    # three of the four products run twice on the tensor cores (bf16 hi and lo parts)
    assert executed == chunks * (2 * Q * Q * N + 2 * (2 * Q * Q * P + 2 * Q * N * P + 2 * Q * N * P))
    elems = 4 * 2048 * 80 * 64
    assert byts == elems * 6 + 4 * 2048 * 1 * N * 2 * 2 + 4 * 2048 * 80 * 2 + 4 * 80 * P * N * 4
