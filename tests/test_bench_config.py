"""bench.py's configuration tables are consistent with each other and with
the repository (no GPU): every workload of the default run exists, every
kernel's source list names real files, and every row of the DRAM traffic
table names a known kernel and workload and parses."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_default_run_covers_every_workload():
    b = load_bench()
    assert set(b.ALL_ORDER) == set(b.WORKLOADS)
    assert b.ALL_ORDER[0] == "decode1"            # the headline line
    for name, wl in b.WORKLOADS.items():
        assert wl["T"] >= 1 and wl["x"] in ("gauss", "clustered"), name


def test_kernel_sources_exist():
    b = load_bench()
    csrc = os.path.join(ROOT, "sparse_moe_transformer_03_b300", "csrc")
    for kernel, files in b.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)
        assert len(b.sources_digest(kernel)) == 16


def test_traffic_table_rows_parse():
    b = load_bench()
    rows = 0
    for ln in open(os.path.join(ROOT, "profiles", "dram_traffic.md")):
        if not ln.startswith("| ") or ln.startswith("| kernel") or ln.startswith("|---"):
            continue
        f = [c.strip() for c in ln.strip().strip("|").split("|")]
        assert f[0] in b.KERNEL_SOURCES, f[0]
        assert f[1] in b.WORKLOADS, f[1]
        assert int(f[2]) > 0 and len(f[3]) == 16
        rows += 1
    assert rows >= 10
