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
