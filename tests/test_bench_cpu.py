"""Host-side helpers of bench.py, without a GPU: the byte models the bench
divides its times by, the compact per-row summary that travels with the
headline line, the lookup of a profiled DRAM traffic figure (used only
while the profiled kernel's sources are unchanged), and the reference arm's
JSON line (the CPU oracle, timed on a small bucket here)."""
import bench


def test_stepwise16_traffic_counts_the_bytes_of_every_step():
    # Units of M (bytes per rank, 2 per 16-bit element). Ring, N = 8:
    # reduce-scatter steps move 8 (2 + 2 in, 4 out), 10 (4 + 2 in, 4 out)
    # x 5 and 8 (4 + 2 in, 2 out) bytes per element of the buffer, the
    # all-gather 7 x (2 + 2): (8 + 50 + 8 + 28) / 2 = 47. Tree, N = 8: levels
    # over 4, 2 and 1 chunk pairs move 4 x 8, 2 x 12 and 1 x 10 bytes per
    # element of a chunk ... the same 94 bytes, 47 M.
    assert bench.stepwise16_traffic("step_ring", 8) == 47
    assert bench.stepwise16_traffic("step_tree", 8) == 47
    # N = 2: one step (2 + 2 in, 2 out) and one copy (2 + 2): (6 + 4) / 2
    assert bench.stepwise16_traffic("step_ring", 2) == 5
    assert bench.stepwise16_traffic("step_tree", 2) == 5
    # N = 4: ring 8 + 10 + 8 and 3 copies; tree 2 x 8 + 1 x 10 and 3 copies
    assert bench.stepwise16_traffic("step_ring", 4) == 19
    assert bench.stepwise16_traffic("step_tree", 4) == 19


def test_rows_summary_keeps_every_row_compact():
    peak = 6774.2
    alg = 2 * bench.NRANKS * bench.COUNT * 4
    ms = alg / (peak * 1e9) * 1e3  # exactly the copy peak
    rows = {
        "ddp_bucket_sync": {
            "direct": {"ms_per_step_eager": 0.7, "ms_per_step_cuda_graph": 0.59, "frac_hbm": 0.9961},
            "three_step": {"ms_per_step_eager": 1.6, "ms_per_step_cuda_graph": 1.7, "frac_hbm": 1.05},
        },
        "fp8_allreduce": {name: {"ms_per_step": 1.5, "frac_hbm": 0.9} for name in
                          ("materialised", "fused_quantisation", "per_hop")},
        "topk_sparse_allreduce": {
            "compress": {"ms": 0.14449, "hbm_gbs_min_bytes": peak * 0.6, "frac_hbm_structure": 0.64,
                         "speculative_share": 1.0, "second_digit_in_pass1_share": 0.95},
            "sparse_allreduce": {"ms": 0.03502, "frac_hbm": 0.903},
        },
    }
    out = bench.rows_summary(rows, {"tree": ms, "ring": 2 * ms}, ms, peak)
    assert out["fused_ring"] == {"ms": round(ms, 4), "frac": 1.0}
    assert out["tree"]["frac"] == 1.0
    assert out["ring_rs_ag"]["frac"] == round((2 * bench.NRANKS + 1) / (2 * bench.NRANKS) / 2, 3)
    assert out["ddp_direct"] == {"ms": 0.59, "frac": 0.996}  # the faster of eager and graph
    assert out["ddp_three_step"]["ms"] == 1.6
    assert set(k for k in out if k.startswith("fp8_")) == {"fp8_materialised", "fp8_fused_quantisation",
                                                          "fp8_per_hop"}
    assert out["topk_compress"] == {"ms": 0.1445, "frac_min_bytes": 0.6, "frac_structure": 0.64,
                                    "speculative_share": 1.0, "second_digit_in_pass1_share": 0.95}
    assert out["sparse_allreduce"] == {"ms": 0.035, "frac": 0.903}
    # rows that did not run are simply absent
    assert set(bench.rows_summary({}, {"tree": ms, "ring": ms}, ms, peak)) == {"fused_ring", "tree", "ring_rs_ag"}


def test_profiled_traffic_only_while_the_sources_match():
    import re

    name = "ar_fused_f32_avg_n8_25MiB.md"
    text = (bench.ROOT / "profiles" / name).read_text(encoding="utf-8")
    recorded = re.search(r"source_hash:\s*([0-9a-f]+)", text).group(1)
    got = bench.profiled_traffic(name)
    if recorded == bench.kernel_source_hash():
        # a figure within 0.2 % of the algorithmic 2 N M bytes
        assert got is not None and abs(got / (2 * bench.NRANKS * bench.COUNT * 4) - 1) < 2e-3
    else:  # the kernel changed since the capture: no traffic is claimed
        assert got is None
    assert bench.profiled_traffic("no_such_profile.md") is None
    # hashed over other sources, the recorded hash no longer matches
    assert bench.profiled_traffic(name, files=bench.FUSED_KERNEL_SOURCES[:1]) is None


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    # the reference arm times the CPU oracle; a small bucket keeps it quick
    import json

    monkeypatch.setattr(bench, "COUNT", 8192)
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(key, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"]) == 0
    lines = [s for s in capsys.readouterr().out.splitlines() if s.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3  # at least 3 warm-up steps
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["dtype"] == "f32"
    assert d["config"]["count_per_rank"] == 8192 and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["kind"] == "oracle" and cb["cores"] == 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # value is the busbw of the timed sample: 2 (N-1)/N x bytes per rank / time
    n = 8192
    assert abs(d["value"] - bench.busbw_gbs(n * 4, d["ms_per_step"] * 1e-3)) < 1e-6 * d["value"]


def test_reference_arm_other_ranks_print_nothing(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
