"""Closed-form traffic, intensity, occupancy and wave counts from the tiling
pages -- TEST INFRASTRUCTURE ONLY (used by tests; the library has its own
scheduling arithmetic and does not import this).

Each function states the passage it restates.  Where a page's arithmetic is
garbled or inconsistent, the function implements the reading given in its
docstring and the tests pin the corrected value.
"""
from __future__ import annotations

import math


# --- "Tiling 策略与内存层次优化" (jonathanding.github.io) -------------------------

def ridge_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """Section "Roofline Model 回顾": ridge = peak FLOP/s / bytes/s."""
    return peak_flops / bandwidth_bytes


def ai_compulsory(M: int, N: int, K: int, elem: int) -> float:
    """Section "Tiling 如何提升算术强度", the first formula: 2MNK / ((MK+KN+MN) * elem).

    This is the compulsory traffic of the whole product (every operand moved
    once).  The page calls it "naive" although its own walk-through (and the
    qian.cx page) use a re-read model; see ``ai_naive_reread``.
    """
    return 2.0 * M * N * K / ((M * K + K * N + M * N) * elem)


def ai_tiled(TM: int, TN: int, elem: int) -> float:
    """Section "Tiling 如何提升算术强度", tiled formula: 2*TM*TN / ((TM+TN) * elem)."""
    return 2.0 * TM * TN / ((TM + TN) * elem)


def naive_per_element(K: int, elem: int) -> tuple[int, int, float]:
    """Walk-through "Step 1": one output reads a row of A and a column of B.

    Returns (FLOPs, bytes read, FLOP/byte) = (2K, 2*K*elem, 1/elem).
    """
    flops = 2 * K
    nbytes = 2 * K * elem
    return flops, nbytes, flops / nbytes


def smem_bytes(BM: int, BN: int, BK: int, elem: int, stages: int) -> int:
    """Section "约束一：Shared Memory 容量": (BM*BK + BK*BN) * elem * stages."""
    return (BM * BK + BK * BN) * elem * stages


def blocks_per_sm_by_smem(smem_per_sm: float, smem_per_block: float) -> int:
    """Same section: floor(SM shared memory / per-block footprint)."""
    return math.floor(smem_per_sm / smem_per_block)


def percent_of_peak(tflops: float, peak: float) -> float:
    """Walk-through summary table: estimated TFLOPS as a percentage of peak."""
    return 100.0 * tflops / peak


# --- "矩阵乘法中的平铺" (qian.cx) ----------------------------------------------

def naive_traffic_bytes(m: int, n: int, k: int, elem: int) -> int:
    """Naive triple loop with no reuse: 2mnk element reads of ``elem`` bytes."""
    return 2 * m * n * k * elem


def ai_naive_reread(elem: int) -> float:
    """(2mnk FLOPs) / (2mnk * elem bytes) = 1/elem; 0.5 for fp16."""
    return 1.0 / elem


def tiled_traffic_elems(m: int, n: int, k: int, b: int) -> float:
    """b x b output tiles: 2*b*k elements per tile, (m/b)(n/b) tiles -> 2mnk/b."""
    return 2.0 * b * k * (m / b) * (n / b)


def ai_output_tiled(b: int, elem: int) -> float:
    """Naive intensity times b, since traffic shrinks by b: 0.5*b FLOP/byte for fp16."""
    return ai_naive_reread(elem) * b


def ksplit_smem_elems(b: int, l: int) -> int:
    """Splitting K into l-length stages: 2*b*l + b*b elements of shared memory."""
    return 2 * b * l + b * b


def ksplit_tile_traffic_elems(b: int, k: int, l: int) -> int:
    """k/l stages of 2*b*l elements: still 2*b*k per output tile (K must divide)."""
    assert k % l == 0
    return (k // l) * 2 * b * l


def compute_bound_tile(peak_flops: float, bandwidth_bytes: float) -> float:
    """0.5*b >= P/B  =>  b >= 2P/B (fp16)."""
    return 2.0 * peak_flops / bandwidth_bytes


def max_b_without_ksplit(S: float, k: int, elem: int) -> float:
    """Reading of the page's capacity bound: the two b x k operand panels,
    2*b*k*elem bytes, must fit in S, so b <= S / (2*k*elem).  (The page prints
    S / (4*k*sizeof); both give single digits at k = 4096, S = 96 KB.)"""
    return S / (2.0 * k * elem)


# --- "寄存器Tiling" (pgsm.cn) ----------------------------------------------------

def register_tile_reads_per_output(K: int, tm: int, tn: int) -> float:
    """Section 1.2: with a tm x tn per-thread tile each output needs K/tn reads of
    A and K/tm reads of B instead of 2K (read as K/8 + K/8 = K/4 for 8x8)."""
    return K / tn + K / tm


def register_budget(tm: int, tn: int, overhead: int) -> int:
    """Section 2.1: tm*tn accumulators + tm A values + tn B values + overhead."""
    return tm * tn + tm + tn + overhead


def occupancy_by_registers(regs_per_thread: int, regs_per_sm: int = 65536, max_threads: int = 2048) -> float:
    """Fraction of the SM's thread slots that fit in its register file.

    Section 1.3 of the page states 128 regs -> 1024 threads (50 %); with the
    65536-register file given on the other two pages the count is 512 (25 %).
    This function uses the register-file arithmetic.
    """
    threads = min(max_threads, regs_per_sm // regs_per_thread)
    return threads / max_threads


# --- "GPU Kernel 的 Tile、Grid、Wave 与 Launch Overhead" (freezetheflame) ---------

def grid(M: int, N: int, BM: int, BN: int) -> tuple[int, int]:
    """grid = (cdiv(M, BM), cdiv(N, BN))."""
    return (-(-M // BM), -(-N // BN))


def regs_per_cta(regs_per_thread: int, warps: int) -> int:
    """regs/thread * warps * 32."""
    return regs_per_thread * warps * 32


def ctas_per_sm_by_registers(regs_per_thread: int, warps: int, regs_per_sm: int = 65536) -> int:
    return regs_per_sm // regs_per_cta(regs_per_thread, warps)


def waves(ctas: int, sms: int, ctas_per_sm: int) -> float:
    """wave count = CTAs / (SMs * CTAs per SM)."""
    return ctas / (sms * ctas_per_sm)


def wave_efficiency(tiles: int, slots: int) -> float:
    """Useful fraction of the last-wave-padded schedule: tiles / (ceil(tiles/slots)*slots)."""
    return tiles / (math.ceil(tiles / slots) * slots)


def tile_load_intensity(BN: int, BK: int, elem: int = 2) -> float:
    """Section "1024²": FLOPs per byte of one (BN + BK) x ... load.

    Reading of the garbled line: loads of BN + BK elements of ``elem`` bytes feed
    BN*BK*2 FLOPs, i.e. 2*BN*BK / ((BN+BK)*elem) -> 21.3 (BN=64) and 25.6 (BN=128)
    for BK = 32, fp16 -- the page's "21" and "26".
    """
    return 2.0 * BN * BK / ((BN + BK) * elem)


def ksweep_traffic_bytes(ctas: int, k_iters: int, BM: int, BN: int, BK: int, elem: int) -> int:
    """Section "2048²": CTAs * K iterations * (BM*BK + BK*BN) * elem bytes.

    The page prints ~16.8 GB for 1024 CTAs x 64 iterations x (64x32 + 32x64)
    fp16; the product is 0.537 GB (and the same for BK = 64 with 32 iterations).
    """
    return ctas * k_iters * (BM * BK + BK * BN) * elem


def tflops_from_time(M: int, N: int, K: int, seconds: float) -> float:
    return 2.0 * M * N * K / seconds / 1e12
