"""Host-side logic of bench.py, on the CPU: the algorithmic bytes behind the
roofline figures, the rule that ncu traffic is reported only for the kernel
sources it was captured from, and the reference arm's JSON line."""
import json
import types

import numpy as np

import bench
import workload as wl


def test_algorithmic_bytes_of_the_benchmark_workload():
    """Byte counts written out from the workload's shapes (8 requests, K = 4,
    S = 32768, 64-byte index rows, top-k 2048, 512-byte K+V rows, 8 query
    heads of 128 dims) with per-request union / miss counts of 3745 / 1271."""
    rec = wl.CONFIGS["cfg2"]
    counts = np.array([[3745, 1271, 1271, 2474]] * 8, np.int64)
    ab = bench.algorithmic_bytes(rec, counts, rec.k_per_req())
    keys = 8 * 32768 * 64
    queries = 8 * 4 * 64
    lists = 4 * 8 * 4 * 2048
    U, M = 8 * 3745, 8 * 1271
    assert ab["select"] == keys + queries + lists == 17_041_408
    kb = ab["kernel_bytes"]
    assert kb["index_score"] == keys + queries
    assert kb["topk"] == 4 * 8 * 4 * 32768 + lists
    assert kb["gather"] == ab["gather"] == M * 512 == 5_206_016
    assert kb["union_probe"] == 2 * lists + 8 * U + 4 * (U + M)
    qo = 2 * 8 * 4 * 8 * (128 + 128)
    assert kb["attn"] == U * 512 + 2 * 32 * 512 + qo + lists
    assert ab["union"] == U and ab["misses"] == M


def test_idle_requests_do_not_count():
    rec = wl.CONFIGS["cfg2"]
    kr = rec.k_per_req().copy()
    kr[3] = 0
    counts = np.zeros((8, 4), np.int64)
    ab = bench.algorithmic_bytes(rec, counts, kr)
    assert ab["select"] == 7 * 32768 * 64 + 7 * 4 * 64 + 4 * 7 * 4 * 2048


def test_ncu_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    summary = tmp_path / "summary.md"
    body = ("# capture\n\n`csrc-sha256: %s`\n\n## k_topk\n- duration: 14.9 us\n"
            "- DRAM read: 4.261888 Mbyte\n- DRAM write: 0.5 Kbyte\n\n"
            "## k_gather<1>\n- DRAM read: 0.531712 Mbyte\n- DRAM write: 5.888 Kbyte\n")
    monkeypatch.setattr(bench, "NCU_SUMMARY", str(summary))
    assert bench.ncu_traffic("topk") is None  # no summary at all
    summary.write_text(body % bench.csrc_hash())
    assert bench.ncu_traffic("topk") == 4_261_888 + 500
    assert bench.ncu_traffic("gather") == 531_712 + 5_888
    assert bench.ncu_traffic("commit") is None  # no section for it
    summary.write_text(body % "0123456789abcdef")
    assert bench.ncu_traffic("topk") is None  # sources changed since the capture


def test_ncu_traffic_scales_by_captured_requests(tmp_path, monkeypatch):
    """A summary captured on a cut of the workload scales each kernel's DRAM
    bytes to the full batch by the file's captured requests, or by a
    section's own count when that kernel was captured on another cut."""
    summary = tmp_path / "summary.md"
    summary.write_text(
        "# capture\n\ncaptured requests: 16\n\n`csrc-sha256: %s`\n\n"
        "## k_index_score_tc<8>\n- DRAM read: 800 Mbyte\n- DRAM write: 40 Mbyte\n\n"
        "## k_topk_row\n- (second capture; captured requests: 48)\n"
        "- DRAM read: 150 Mbyte\n- DRAM write: 3 Mbyte\n" % bench.csrc_hash())
    monkeypatch.setattr(bench, "NCU_SUMMARY", str(summary))
    assert bench.ncu_traffic("index_score", full_requests=128) == 8 * 840_000_000
    assert bench.ncu_traffic("topk", full_requests=96) == 2 * 153_000_000
    assert bench.ncu_traffic("topk") == 153_000_000  # no scaling without a batch


def test_csrc_hash_is_stable():
    h = bench.csrc_hash()
    assert h == bench.csrc_hash() and len(h) == 16
    int(h, 16)


def test_reference_arm_line(capsys):
    """The reference arm times the oracle on one request's round per step, on
    a pool of one process per host core, and prints the contract's line with
    impl = reference and the native arm's config object."""
    args = types.SimpleNamespace(workload="cfg1", steps=1, warmup=0, batch=0)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "query-tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == bench.host_cores() >= 1
    assert line["config"] == bench.workload_config(wl.CONFIGS["cfg1"])


def test_reference_arm_under_two_ranks():
    """Launched as the contract launches N > 1 (torchrun, one process per
    rank), the reference arm prints one line, from rank 0; the other rank
    exits 0 without work."""
    import os
    import socket
    import subprocess
    import sys
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "cfg1"]
    p = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    # one pool over the node's cores, not one per rank: labelled as such
    assert line["per_rank"] is False and line["scaling"] == "none"
    assert "does not grow with n_gpus" in line["reference_scope"]
