"""The pages' worked byte/FLOP/occupancy/wave counts (tests/golden/page_numbers.json)."""
import json
import os

import pytest

from oracle import perfmodel as pm

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
ENTRIES = {e["id"]: e for e in GOLDEN["entries"]}


def close(got, e):
    want = e["value"]
    if "decimals" in e:   # compare at the precision the page prints
        assert [round(g, d) for g, d in zip(got, e["decimals"])] == want, (e["id"], got, want)
        return
    if isinstance(want, list):
        assert len(got) == len(want)
        for g, w in zip(got, want):
            close(g, {**e, "value": w})
        return
    if "abs" in e:
        assert abs(got - want) <= e["abs"], (e["id"], got, want)
    else:
        assert abs(got - want) <= e.get("rel", 0.0) * abs(want), (e["id"], got, want)


def compute(eid):
    i = ENTRIES[eid]["inputs"]
    if eid == "ridge_a100":
        return pm.ridge_point(i["peak"], i["bw"])
    if eid == "tiled_ai_128_fp16":
        return pm.ai_tiled(i["TM"], i["TN"], i["elem"])
    if eid == "naive_element_flops":
        return pm.naive_per_element(i["K"], i["elem"])[0]
    if eid == "naive_element_bytes":
        return pm.naive_per_element(i["K"], i["elem"])[1]
    if eid == "naive_element_ai":
        return pm.naive_per_element(i["K"], i["elem"])[2]
    if eid in ("smem_128_128_32_2stage", "smem_256_256_64_3stage"):
        return pm.smem_bytes(i["BM"], i["BN"], i["BK"], i["elem"], i["stages"])
    if eid == "blocks_per_sm_a100":
        return pm.blocks_per_sm_by_smem(i["smem_kb"], i["block_kb"])
    if eid == "ladder_percent":
        return [pm.percent_of_peak(t, i["peak"]) for t in i["tflops"]]
    if eid == "naive_ai_qian":
        return pm.ai_naive_reread(i["elem"])
    if eid == "v100_p_over_b":
        return pm.ridge_point(i["peak"], i["bw"])
    if eid == "v100_b_threshold":
        return pm.compute_bound_tile(i["peak"], i["bw"])
    if eid == "register_tile_reduction":
        return 2 * i["K"] / pm.register_tile_reads_per_output(i["K"], i["tm"], i["tn"])
    if eid == "register_budget_range":
        return [pm.register_budget(i["tm"], i["tn"], o) for o in i["overhead"]]
    if eid == "regs_per_worker":
        return pm.regs_per_cta(i["regs"], i["warps"])
    if eid in ("workers_per_sm_128", "workers_per_sm_200"):
        return pm.ctas_per_sm_by_registers(i["regs"], i["warps"])
    if eid == "waves":
        return [pm.waves(c, i["sms"], i["per_sm"]) for c in i["ctas"]]
    if eid == "grid_counts":
        return [list(pm.grid(n, n, b, b)) for n, b in i["shapes"]]
    if eid == "tile_load_intensity":
        return [pm.tile_load_intensity(bn, i["BK"], i["elem"]) for bn in i["BN"]]
    if eid == "ksweep_traffic_gb":
        t32 = pm.ksweep_traffic_bytes(i["ctas"], i["iters"][0], i["BM"], i["BN"], i["BK"][0], i["elem"])
        t64 = pm.ksweep_traffic_bytes(i["ctas"], i["iters"][1], i["BM"], i["BN"], i["BK"][1], i["elem"])
        assert t32 == t64
        return t32 / 1e9
    if eid == "rtx4070s_4096_tflops":
        return pm.tflops_from_time(i["M"], i["M"], i["M"], i["seconds"])
    if eid == "cuda_tile_64_grid":
        return list(pm.grid(i["M"], i["N"], i["BM"], i["BN"]))
    raise KeyError(eid)


@pytest.mark.parametrize("eid", sorted(ENTRIES))
def test_page_number(eid):
    got = compute(eid)
    if eid == "grid_counts" or eid == "cuda_tile_64_grid":
        assert got == ENTRIES[eid]["value"]
    else:
        close(got, ENTRIES[eid])


def test_k_split_keeps_traffic():
    # "矩阵乘法中的平铺": k/l stages of 2bl elements still move 2bk per tile
    for l in (8, 16, 64, 256):
        assert pm.ksplit_tile_traffic_elems(128, 4096, l) == 2 * 128 * 4096
    assert pm.tiled_traffic_elems(1024, 2048, 4096, 128) == 2 * 1024 * 2048 * 4096 / 128
    assert pm.ai_output_tiled(128, 2) == 64.0
    assert pm.ksplit_smem_elems(128, 64) == 2 * 128 * 64 + 128 * 128


def test_capacity_bound_single_digits():
    # "矩阵乘法中的平铺": at k = 4096, S ~ 96 KB, fp16, b without K-splitting is single digits
    assert 1 <= pm.max_b_without_ksplit(96 * 1024, 4096, 2) < 10


def test_compulsory_intensity_large_k():
    # "Tiling 策略与内存层次优化": 2MNK/((MK+KN+MN) e) -> 2K/e as M, N >> K
    v = pm.ai_compulsory(10 ** 7, 10 ** 7, 64, 2)
    assert abs(v - 2 * 64 / 2) / 64 < 1e-4
    # 4096^3 bf16 in, fp32 out (traffic of the headline product)
    assert abs(2 * 4096 ** 3 / ((2 * 4096 ** 2) * 2 + 4096 ** 2 * 4) - 1024) < 1e-9


def test_occupancy_register_arithmetic():
    # 65536 registers / 128 per thread = 512 threads of 2048 = 25 %
    assert pm.occupancy_by_registers(128) == 0.25
    assert pm.occupancy_by_registers(32) == 1.0
