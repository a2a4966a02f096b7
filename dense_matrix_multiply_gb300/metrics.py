"""Host-side GEMM accounting: FLOPs, bytes, peaks and the per-warp "beat".

Pure arithmetic on shapes, clocks and times; no GPU is touched. The formulas are
the pages' own:
  * FLOPs = 2*M*N*K, one FMA counted as two operations ("SGEMM measured and the
    three ledgers", K3 step 3; "Chapter 5 Operators and Runtime", section 5.2.1).
  * minimum bytes = elt*(M*K + K*N + M*N), each matrix crossing the memory
    interface once; tiled bytes = elt*(M*K*ceil(N/bn) + K*N*ceil(M/bm) + M*N) when
    every output tile reads its own inputs and no cache helps ("K1 walkthrough:
    the GEMM resource ledger", section 2; "Chapter 5", section 5.2.2, example 5-3).
  * per-tile working set = in_elt*(m*k + k*n) + acc_elt*m*n ("Chapter 5",
    example 5-3).
  * FP32 SIMT peak = SMs * 128 lanes * 2 * clock, and the beat
    32 * SMs * clock * t / (M*N*K), cycles per warp-round ("SGEMM measured and the
    three ledgers", section 2 and K3 step 6).
"""

from __future__ import annotations

import math


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def min_bytes(M: int, N: int, K: int, elt: int) -> int:
    return elt * (M * K + K * N + M * N)


def tiled_bytes(M: int, N: int, K: int, elt: int, bm: int, bn: int) -> int:
    return elt * (M * K * math.ceil(N / bn) + K * N * math.ceil(M / bm) + M * N)


def tile_working_set(m: int, n: int, k: int, in_elt: int = 2, acc_elt: int = 4) -> int:
    return in_elt * (m * k + k * n) + acc_elt * m * n


def simt_fp32_peak(sms: int, clock_hz: float, lanes_per_sm: int = 128) -> float:
    """FLOP/s of FFMA on every FP32 lane of every SM at the given clock."""
    return sms * lanes_per_sm * 2 * clock_hz


def flops_per_s(M: int, N: int, K: int, seconds: float) -> float:
    return gemm_flops(M, N, K) / seconds


def beat(sms: int, clock_hz: float, seconds: float, M: int, N: int, K: int) -> float:
    """Cycles per warp-round: each SM retires 32*4 FMA lanes per cycle at best, so a
    perfect FP32 kernel on 128-lane SMs sits at 0.25."""
    return 32 * sms * clock_hz * seconds / (M * N * K)


def wave_count(tiles: int, slots: int) -> float:
    """Tiles divided by concurrently resident tiles (SMs x CTAs per SM)."""
    return tiles / slots


def wave_efficiency(tiles: int, slots: int) -> float:
    """Useful fraction of the last-wave-rounded schedule: tiles / (ceil(waves) * slots)."""
    if tiles == 0:
        return 1.0
    return tiles / (math.ceil(tiles / slots) * slots)


def fp8_rowscale_traffic(M: int, K: int, N: int, tile_n: int, in_elt: int = 2, q_elt: int = 1,
                         w_elt: int = 1, out_elt: int = 2, tile_m: int = 128) -> dict:
    """Bytes moved by a row-scaled FP8 projection when every output tile reads
    its operands independently ("Chapter 5 Operators and Runtime", example 5-8).
    Both schemes first read the whole input once to find each row's scale.
    separate: write the FP8 input once, then every column block re-reads it.
    fused: every column block re-reads the 16-bit input and quantises locally.
    Both: every row block reads the whole weight matrix; the output is written
    once."""
    col_blocks = -(-N // tile_n)
    row_blocks = -(-M // tile_m)
    a_in, a_q = M * K * in_elt, M * K * q_elt
    separate_in = a_in + a_q + col_blocks * a_q
    fused_in = a_in + col_blocks * a_in
    w_out = row_blocks * K * N * w_elt + M * N * out_elt
    return {"separate_input": separate_in, "fused_input": fused_in, "weights_output": w_out,
            "separate_total": separate_in + w_out, "fused_total": fused_in + w_out}
