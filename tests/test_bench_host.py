"""Host-side bookkeeping of the benchmark (no GPU): the code digest that keys the
profiled DRAM traffic, and the accounting behind the roofline figures."""
import bench
import moe_workloads as mw


def test_code_digest_ignores_comments_only():
    src = "int f(int a) {\n    return a + 1;  // one more\n}\n"
    commented = "/* header\n   text */\n" + src.replace("// one more", "// a longer note") + "\n\n"
    changed = src.replace("a + 1", "a + 2")
    assert bench.code_digest(src) == bench.code_digest(commented)
    assert bench.code_digest(src) != bench.code_digest(changed)


def test_profiled_traffic_unknown_stage_is_none():
    assert bench.profiled_traffic("no_such_stage", mw.T8192.name) is None


def test_alu_partials_counts_every_block_scale():
    # gate/up: two f x d matrices over d/32 blocks; down: one d x f matrix over f/32
    cfg = mw.T8192
    R = cfg.T * cfg.K
    want = R * 2 * cfg.f * (cfg.d // 32) + R * cfg.d * (cfg.f // 32)
    assert bench.alu_partials(cfg, R) == want


def test_profiled_traffic_entries_name_real_sources():
    import os
    for (stage, workload), rec in bench.PROFILED_TRAFFIC.items():
        assert workload in mw.CONFIGS, workload
        assert os.path.exists(os.path.join(bench.ROOT, rec["source"])), rec["source"]
        assert len(rec["code_sha256_16"]) == 16 and rec["bytes"] > 0


def test_layer_accounting_q8_1_bytes_per_layout():
    """Activations cost 1.125 bytes a value in the (d, s) layout and 1.25 in D2S6
    (Q2_K): the quantize-scatter bytes differ by exactly R*d*0.125."""
    acc = {}
    for cfg in (mw.T2048_Q2, mw.T2048_Q2K):
        R = cfg.T * cfg.K
        stages, _, _ = bench.layer_accounting(cfg, 512, 1 << 20, R)
        acc[cfg.wtype] = stages["quantize_scatter"][0]
    cfg = mw.T2048_Q2K
    assert acc[mw.Q2_K] - acc[mw.Q2_0] == cfg.T * cfg.K * cfg.d * 0.125
