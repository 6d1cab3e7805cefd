"""The roofline numerator: algorithmic bytes per pass or step, as bench.py
counts them, against the figures worked out by hand from the layouts
(every input read once, y written once, state and carry read and written
once)."""
import bench
import synth

W = synth.workloads()


def test_siso_prefill_bytes():
    b = bench.workload_bytes(W["siso_b8_l4096"])
    # per token and head: x 128, B 256, C 256, theta 128, dt + lam 4, y 256 (f32)
    assert b["per_token_head"] == 1028
    th = 8 * 4096 * 32
    state = 8 * 32 * 128 * 64 * 4 * 2
    carry = 8 * 32 * (128 + 64) * 2 * 2
    assert b["per_unit_of_work"] == th * 1028 + state + carry == 1_094_909_952


def test_mimo_prefill_bytes():
    # x 512, B 512, C 512, theta 64, dt + lam 4, y 1024
    assert bench.workload_bytes(W["mimo4_b8_l4096"])["per_token_head"] == 2628


def test_variants_change_only_their_part():
    # one B/C group for 32 heads: B and C cost 2 * 256 / 32 per token and head
    assert bench.workload_bytes(W["siso_g1_b8_l4096"])["per_token_head"] == 1028 - 512 + 16
    # bf16 y: 128 instead of 256
    assert bench.workload_bytes(W["siso_ybf16_b8_l4096"])["per_token_head"] == 1028 - 128
    # Mamba-2 special case: no theta (128) and no lam (2) read
    assert bench.workload_bytes(W["mamba2_b8_l4096"])["per_token_head"] == 1028 - 130
    # the raw-input workload reads the same bytes (dt_bias is per head only)
    assert bench.workload_bytes(W["siso_prologue_b8_l4096"])["per_token_head"] == 1028


def test_decode_step_bytes():
    b = bench.workload_bytes(W["decode_siso_b256"])
    units = 256 * 32
    state = units * 64 * 128 * 4 * 2  # f32 state read and written
    assert b["state"] == state == 536_870_912
    # inputs x 128 + B 256 + C 256 + theta 128 + dt + lam 4, carry read and written, y f32
    assert b["per_unit_of_work"] == state + units * 772 + units * 384 * 2 + units * 256 == 551_583_744


def test_contraction_flops_against_hand_derived_figures():
    """Tensor-core work of the chunked form: 2QN + 2QP + 4NP per token and
    head for SISO (Q 64, N 128, P 64: 57,344, i.e. 60.1 GFLOP for the batch
    8 x 4096 x 32-head pass); 2QR^2 N + 2QR^2 P + 4RNP for MIMO at Q 16, R 4,
    N 64; and the issued MMAs with their hi/lo operand pairs (three products
    for a rotated operand, two for S' and for C R)."""
    w = synth.workloads()
    f = bench.contraction_flops(w["siso_b8_l4096"])
    assert f["per_token_head"] == 57344
    assert f["algorithmic"] == 57344 * 8 * 4096 * 32
    # per 64-token chunk: MMA 1 3 x 2*64*64*128, MMA 2 2 x 2*64*64*64, MMA 3 2 x 2*64*64*128, MMA 4 3 x 2*128*64*64
    per_chunk = 3 * 1048576 + 2 * 524288 + 2 * 1048576 + 3 * 1048576
    assert f["issued"] == per_chunk * 8 * 4096 * 32 // 64
    m = bench.contraction_flops(w["mimo4_b8_l4096"])
    assert m["per_token_head"] == 2 * 16 * 16 * 64 + 2 * 16 * 16 * 64 + 4 * 4 * 64 * 64
    r = bench.contraction_flops(w["mamba2_b8_l4096"])  # real state: B and C exact in f16, one product each
    per_chunk_re = 1048576 + 2 * 524288 + 1048576 + 2 * 1048576
    assert r["issued"] == per_chunk_re * 8 * 4096 * 32 // 64
    assert bench.contraction_flops(w["decode_siso_b256"]) == {}
