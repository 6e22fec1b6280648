"""The byte and flop accounting bench.py reports its rooflines with, checked
against counts done by hand (no GPU)."""
import torch

import bench
from gated_deltanet_linear_04_gb300 import workloads as wl


def test_decode_bytes_of_the_batched_decode_workload():
    d = wl.WORKLOADS["decode_b128"].dims
    by = bench.decode_bytes(d)
    assert by["state_rw"] == 2 * 128 * 32 * 128 * 128 * 4          # 536.9 MB
    C = 2 * 16 * 128 + 32 * 128
    assert by["conv_state_rw"] == 2 * 128 * 3 * C * 2
    assert sum(by.values()) == 552681728                           # the decode roofline's bytes


def test_chunk_mma_flops_counts_each_product():
    d = wl.WORKLOADS["prefill_t8192"].dims                          # Dk = Dv = 128
    C = 64
    products = [(2 * C, C, 128),      # [K;Q] K^T
                (C, C, 128),          # U = T diag(beta) V
                (C, C, 128),          # W = T diag(beta gamma) K
                (C, 128, 128),        # D = U - W S0^T
                (C, 128, 128),        # S0 part of Y
                (128, 128, C),        # state update D^T P
                (C, C, 128)]          # intra-chunk part of Y
    assert bench.chunk_mma_flops(d) == sum(2 * m * n * k for m, n, k in products)


def test_active_chunks_counts_chunks_with_a_valid_step():
    T, B = 300, 5
    lens = torch.tensor([0, 1, 64, 65, 300])
    mask = wl.right_padded_mask(lens, T)
    assert bench.active_chunks(mask, T, B) == 0 + 1 + 1 + 2 + 5
    assert bench.active_chunks(None, T, B) == B * 5
    holes = torch.zeros((1, T), dtype=torch.uint8)
    holes[0, 130] = 1                                               # one valid step in chunk 2
    assert bench.active_chunks(holes, T, 1) == 1


def test_profiled_traffic_only_for_the_profiled_source(monkeypatch, tmp_path):
    """roofline.traffic comes from a committed profile summary only while the
    profiled kernel source hashes to the value recorded in it, else null."""
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text("source_hash: abcdef0123456789   (note)\n"
                                                "dram_bytes_per_launch: 495584000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda *names: "abcdef0123456789")
    assert bench.profiled_traffic("k.md", ["decode.cu"]) == 495584000.0
    monkeypatch.setattr(bench, "source_hash", lambda *names: "0" * 16)
    assert bench.profiled_traffic("k.md", ["decode.cu"]) is None
    assert bench.profiled_traffic("missing.md", ["decode.cu"]) is None


def test_fp32_peak_from_unit_counts_and_clock():
    # 152 SMs x 128 FP32 lanes x one FMA (2 flops) per clock at 2070 MHz
    assert abs(bench.fp32_peak_tflops(2070.0) - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
    assert 80.0 < bench.fp32_peak_tflops(2070.0) < 81.0


def test_conv_bytes_of_the_prefill_workload():
    d = wl.WORKLOADS["prefill_t8192"].dims
    C = 2 * 16 * 128 + 32 * 128                                     # 8192 channels
    n = d.B * d.T
    # qkv in and q/k/v out (bf16) per token, the taps, conv_state in and out
    assert bench.conv_bytes(d, n) == n * C * 2 * 2 + C * 4 * 2 + 2 * 3 * C * 2
    # padded tokens read nothing but still get their zero outputs written
    assert bench.conv_bytes(d, 0) == n * C * 2 + C * 4 * 2 + 2 * 3 * C * 2


def test_oracle_prefill_rate_reports_a_bounded_sample():
    """The CPU baseline of a prefill entry: whole heads at the workload's T,
    the tokens/s figure scaled from the heads it ran to all Hv heads."""
    w = wl.Workload("small", 9, wl.Dims(B=2, T=96, Hk=2, Hv=4, Dk=32, Dv=32), ragged=True, len_lo=10,
                    len_hi=96)
    r = bench.oracle_prefill_rate(w, heads_per_row=2)
    lens = wl.workload_lengths(w)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["cores"] >= 1
    steps = int(lens.sum()) * 2
    assert "(%d valid head-steps)" % steps in r["sample"]
    assert abs(r["value"] - steps / 4 / r["seconds"]) <= 0.06 * r["value"] + 1.0
    rv = bench.oracle_prefill_rate(w, heads_per_row=1, vec=True)
    assert rv["value"] > 0 and "per-channel" in rv["sample"]


def test_backward_chunk_flops_product_by_product():
    # every product of the chunked backward (M, N, K) at C = 64, Dk = Dv = 128,
    # 2 flops per multiply-add, counted one by one
    d = wl.Dims(B=1, T=64, Hk=1, Hv=1, Dk=128, Dv=128)
    C, D = 64, 128
    products = [
        # the forward with chunk records
        (2 * C, C, D), (C, C, D), (C, C, D), (C, D, D), (C, D, D), (C, C, D), (D, D, C),
        # chain images: [K;Q] K^T, Wb, dY^T P, (dY^T P) T, Cq
        (2 * C, C, D), (D, C, C), (D, C, C), (D, C, C), (D, D, C),
        # reverse chain: dZ^T += G Wb^T, G += dZ^T diag(beta) (-gamma K)
        (D, C, D), (D, D, C),
        # gradients I: [K;Q] K^T, S0 [gamma K; gamma Q]^T, [dY; dZ] D^T
        (2 * C, C, D), (D, 2 * C, D), (2 * C, C, D),
        # gradients II: S0^T [dY; dZ]^T, G^T D^T, K^T [dPM; H + H^T]^T, Q^T dPM
        (D, 2 * C, D), (D, C, D), (D, 2 * C, C), (D, C, C),
    ]
    assert bench.backward_chunk_mma_flops(d) == sum(2 * m * n * k for m, n, k in products)
