"""Host arithmetic of the benchmark, on CPU: the algorithmic bytes of each
kernel, and the roofline block's use of a recorded ncu traffic figure only
while the CUDA sources keep the digest it was captured on."""
import pytest

import bench
import workloads

# Algorithmic bytes per step in MB, all ranks, as tabulated for the four
# workloads: 16-bit input; codes of 1 B (FP8, INT8) or 0.5 B (INT4); block
# metadata of 1 B per block (TACO) or 4 B per block (INT8 sym: FP32 scale;
# asym: fp16 scale and fp16 zero-point); the FP32 sum of K2 / K3.
TABLE_MB = {
    "gpt_tp": {"K1": 807.4, "K2": 404.8, "K3": 168.0, "K4": 100.9},
    "qwen_grad": {"K1": 504.0, "K2": 336.2, "K3": 209.9, "K4": 126.0},
    "equarx_int8": {"K1": 3288.3, "K2": 1677.7, "K3": 679.5, "K4": 411.0},
    "flash_int4": {"K1": 1359.0, "K2": 553.6, "K3": 337.6, "K4": 203.4},
}


@pytest.mark.parametrize("name", sorted(TABLE_MB))
def test_algorithmic_bytes_match_the_table(name):
    alg = bench.algorithmic_bytes(workloads.WORKLOADS[name])
    for k, mb in TABLE_MB[name].items():
        assert alg[k] / 1e6 == pytest.approx(mb, abs=0.051), k
    # the fused reduce + requant reads the shards and writes the gather codes:
    # the two-call path's bytes less the FP32 sum written and read back
    E = workloads.WORKLOADS[name].elems_per_rank
    assert alg["K23"] == pytest.approx(alg["K2"] + alg["K3"] - 8 * E)


def test_roofline_takes_traffic_only_for_its_digest(monkeypatch):
    w = workloads.WORKLOADS["qwen_grad"]
    alg = bench.algorithmic_bytes(w)
    kern = {"K1": {"ms": 0.1}}
    entry = bench.NCU_TRAFFIC[("taco_compress", w.name)]
    monkeypatch.setattr(bench, "_src_digest", lambda: entry["src"])
    r = bench._roofline(w, kern, alg, (6000.0, "measured"))
    assert r["traffic"] == entry["bytes"]
    assert r["achieved"] == pytest.approx(alg["K1"] / 1e-4 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)
    assert r["peak_source"] == "measured hbm_gbs" and r["bound"] == "hbm"
    monkeypatch.setattr(bench, "_src_digest", lambda: "0" * 16)
    assert bench._roofline(w, kern, alg, (6000.0, "measured"))["traffic"] is None


@pytest.mark.parametrize("key", sorted(bench.NCU_TRAFFIC))
def test_recorded_traffic_is_near_the_algorithmic_bytes(key):
    # K1 reads its input once and writes its codes once; part of the codes can
    # still be dirty in L2 when it ends, so DRAM traffic sits a little below the
    # algorithmic bytes, never far above them (that would mean re-reads)
    alg = bench.algorithmic_bytes(workloads.WORKLOADS[key[1]])["K1"]
    t = bench.NCU_TRAFFIC[key]["bytes"]
    assert 0.85 * alg < t <= 1.02 * alg
