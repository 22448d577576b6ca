"""bench.py's host logic on CPU: the algorithmic-traffic model (the missed rows'
host reads and slot writes are charged to the kernel that copies them, totals do
not depend on which one that is), the code hash that keys the committed ncu
figures, the package's Belady MIN against the oracle's, the reference arm's
JSON line, and the attention timeline derived from two hs_stats snapshots."""
import os

import numpy as np

import workload as wl


def test_pulled_rows_are_charged_to_the_copying_kernel():
    import bench
    w = wl.WORKLOADS["batch16_32k"]
    n_ctx = w.contexts() + 5
    a = bench.algorithmic_bytes(w, n_ctx, 700.0, resolve_pulls=False)
    b = bench.algorithmic_bytes(w, n_ctx, 700.0, resolve_pulls=True)
    moved = 700.0 * w.row_bytes
    assert b["link"]["select"] - a["link"]["select"] == moved
    assert a["link"]["attention"] - b["link"]["attention"] == moved
    assert b["hbm"]["select"] - a["hbm"]["select"] == moved
    for kind in ("hbm", "link"):
        assert np.isclose(sum(a[kind].values()), sum(b[kind].values()))
    # the index scan reads every key once (it dominates the select kernel's bytes);
    # the attention every selected row once (with RESOLVE copying the misses,
    # nothing else)
    assert a["hbm"]["select"] >= float((n_ctx * w.d_idx).sum()) + w.n_requests * w.d_idx
    k_eff = np.minimum(w.top_k, n_ctx).sum()
    assert b["hbm"]["attention"] == float(k_eff) * (w.row_bytes + 4) + w.n_requests * w.h_q * (w.d_qk + w.d_v) * 2


def test_who_pulls_follows_the_library_rule():
    import bench
    assert bench.resolve_pulls(1, False)
    assert bench.resolve_pulls(0, True)          # latent rows: always RESOLVE
    assert not bench.resolve_pulls(0, False)
    assert not bench.resolve_pulls(2, False)     # the default: the attention kernel


def test_code_hash_ignores_comments_only(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;   // store\n}\n")
    h = bench.code_hash(str(a))
    a.write_text("// a different header\n\n__global__ void k(int* p) {\n  p[0] = 1;\n}\n// tail\n")
    assert bench.code_hash(str(a)) == h
    a.write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n")
    assert bench.code_hash(str(a)) != h



def test_library_belady_equals_the_oracle():
    # the package's host-side MIN (used by the benchmark's policy-floor leg) and
    # the oracle's, written separately, agree on random set traces
    from oracle import belady_misses as oracle_min
    from tiered_kv_cache_int8_gb300.analysis import belady_misses as lib_min
    rng = np.random.default_rng(31)
    for _ in range(300):
        k = int(rng.integers(1, 7))
        B = k + int(rng.integers(0, 6))
        n_pos = int(rng.integers(k, 40))
        trace = [sorted(rng.choice(n_pos, size=k, replace=False).tolist()) for _ in range(int(rng.integers(1, 20)))]
        assert lib_min(trace, B) == oracle_min(trace, B)


def _optimal_misses(refs, B):
    """Fewest misses over every eviction choice (exhaustive; tiny traces only)."""
    from functools import lru_cache

    @lru_cache(maxsize=None)
    def best(i, cached):
        if i == len(refs):
            return 0
        p = refs[i]
        if p in cached:
            return best(i + 1, cached)
        if len(cached) < B:
            return 1 + best(i + 1, cached | {p})
        return 1 + min(best(i + 1, (cached - {q}) | {p}) for q in cached)
    return best(0, frozenset())


def test_library_belady_equals_an_exhaustive_optimum():
    # pinned on its own, not only against the oracle: on tiny step-serialised
    # traces MIN's count equals the minimum over every possible eviction choice
    from tiered_kv_cache_int8_gb300.analysis import belady_misses as lib_min
    rng = np.random.default_rng(77)
    for _ in range(150):
        k = int(rng.integers(1, 4))
        B = k + int(rng.integers(0, 3))
        n_pos = int(rng.integers(k, 8))
        trace = [sorted(rng.choice(n_pos, size=k, replace=False).tolist()) for _ in range(int(rng.integers(1, 7)))]
        refs = tuple(p for s in trace for p in s)
        assert lib_min(trace, B) == _optimal_misses(refs, B)


def test_reference_arm_line_on_cpu():
    # the reference arm (the oracle, timed on host cores) prints one JSON line with
    # the contract's keys; tiny workload, a few steps
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["metric"] and d["unit"] == "layer-steps/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_bench_names_resolve():
    # every module-level name bench.py uses is defined (catches a helper lost in an edit)
    import ast
    import builtins
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    tree = ast.parse(open(os.path.join(root, "bench.py")).read())
    defined = {n.name for n in tree.body if isinstance(n, (ast.FunctionDef, ast.ClassDef))}
    for n in tree.body:
        if isinstance(n, ast.Assign):
            defined |= {t.id for t in n.targets if isinstance(t, ast.Name)}
    for n in ast.walk(tree):   # imports, also those inside functions
        if isinstance(n, (ast.Import, ast.ImportFrom)):
            defined |= {(a.asname or a.name).split(".")[0] for a in n.names}
    called = {c.func.id for c in ast.walk(tree) if isinstance(c, ast.Call) and isinstance(c.func, ast.Name)}
    local = {a.arg for f in ast.walk(tree) if isinstance(f, (ast.FunctionDef, ast.Lambda)) for a in f.args.args}
    local |= {t.id for a in ast.walk(tree) if isinstance(a, ast.Assign) for t in a.targets if isinstance(t, ast.Name)}
    local |= {f.name for f in ast.walk(tree) if isinstance(f, ast.FunctionDef)}
    missing = sorted(c for c in called if c not in defined and c not in local and not hasattr(builtins, c))
    assert not missing, missing


def test_attention_timeline_from_two_snapshots():
    # the exposed link time is the host stages' waits beyond the mean wait of an
    # HBM-only stage; the balance figures come from the later snapshot; latent rows
    # (no counts) report nothing
    import bench
    keys = ("att_host_wait_ns", "att_host_stages", "att_hbm_wait_ns", "att_hbm_stages", "att_last_span_ns",
            "att_last_median_ns")
    st0 = dict(zip(keys, (1000, 1, 500, 1, 7, 7)))
    st1 = dict(zip(keys, (1000 + 4 * 3000, 1 + 4, 500 + 10 * 1000, 1 + 10, 60000, 50000)))
    t = bench.attention_timeline(st0, st1, n_launch=2, n_cta=2)
    assert t["host_stage_wait_us"] == 3.0 and t["hbm_stage_wait_us"] == 1.0
    # 4 host stages waited 12 us where HBM-only stages would have taken 4 us: 8 us
    # over 2 launches x 2 CTAs
    assert t["link_exposed_us_per_cta_layer"] == 2.0
    assert t["host_stages_per_cta_layer"] == 1.0
    assert t["last_launch_span_us"] == 60.0 and t["span_over_median"] == 1.2
    assert bench.attention_timeline(st1, st1, 2, 2) is None
