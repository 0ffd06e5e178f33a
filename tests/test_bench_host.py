"""Host logic of bench.py: the algorithmic bytes and FLOPs it divides by, the
paths and kernels it times, the rotating input sets, and the rule that an ncu
summary's traffic is used only while the kernel's sources are unchanged."""
import numpy as np
import pytest

import bench
import workloads as W


def test_algorithmic_bytes_by_hand_for_the_decode_shape():
    cfg = W.CONFIGS["decode"]
    ends = np.array([8192, 65536, 1000], np.int64)    # 1000 < K: fewer winners than K
    R = cfg.rows
    S, K, H, D = cfg.S, cfg.K, cfg.H, cfg.D
    b = bench.algorithmic_bytes(cfg, ends)
    logits = 4 * (8192 + 65536 + 1000)
    assert b["shard_topk_pack"] == logits + R * 8 * S * K
    assert b["merge_topk_stable"] == R * (8 * S * K + 4 * K)
    assert b["convert_index_compact"] == R * (4 * K + 4 * K + 4 * S * K + 4 * S)
    assert b["indexer_fused"] == logits + R * (8 * K + 4 * S * K + 4 * S)
    assert b["lse_combine"] == R * (S * H * D * 2 + S * H * 4 + H * D * 2 + H * 4)
    assert b["slot_mapping"] == R * (4 + 4 + 4 * S)               # row r is request r
    sel = 2048 + 2048 + 1000
    assert bench.selected(cfg, ends) == sel
    assert b["sparse_mla_decode"] == sel * (4 + 1152) + R * S * (H * 1152 + 4 + H * 1028)
    assert bench.attention_flops(cfg, ends) == 2 * H * sel * (576 + 512)


def test_prefill_write_side_counts_the_request_word():
    cfg = W.CONFIGS["prefill"]
    _, ends = W.row_ranges(cfg)
    assert bench.algorithmic_bytes(cfg, ends)["slot_mapping"] == cfg.rows * (4 + 4 + 4 + 4 * cfg.S)


def test_paths_kernels_metrics():
    dec, tiny = W.CONFIGS["decode"], W.CONFIGS["tiny"]
    assert bench.kernels_for(dec, "fused") == ("indexer_fused", "lse_combine")
    assert bench.kernels_for(tiny, "fused") == ("indexer_fused",)          # no heads: no combine
    assert bench.kernels_for(dec, "attention") == ("indexer_fused", "sparse_mla_decode",
                                                   "lse_combine")
    assert bench.kernels_for(dec, "write_slots") == ("slot_mapping",)
    assert bench.metric_for("fused") == (bench.METRIC, "rows/s")
    assert bench.metric_for("write_slots")[1] == "tokens/s"
    assert bench.dtype_for("write_slots") == "i32" and bench.dtype_for("steps") == "f32"
    for k in ("indexer_fused", "lse_combine", "shard_topk_pack", "merge_topk_stable",
              "convert_index_compact", "slot_mapping", "sparse_mla_decode"):
        assert k in bench.KERNEL_SOURCES


@pytest.mark.parametrize("name", sorted(W.CONFIGS))
def test_rotating_sets_exceed_l2(name):
    cfg = W.CONFIGS[name]
    n = bench.replicas_for(cfg)
    assert 2 <= n <= 8
    assert n * bench.set_bytes(cfg) > 2.5 * bench.L2_BYTES or n == 8


def test_profile_traffic_only_while_sources_match(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    h = bench.kernel_source_hash("indexer_fused")
    (tmp_path / "profiles" / "indexer_fused_decode.md").write_text(
        f"# summary\n\nsource_sha256_16: {h}\ndram_bytes_per_launch: 10274816\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: h)
    assert bench.profiled_traffic("indexer_fused", "decode") == 10274816
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.profiled_traffic("indexer_fused", "decode") is None
    assert bench.profiled_traffic("no_such_kernel", "decode") is None


def test_committed_profiles_name_their_sources():
    """Every committed kernel summary states the source hash and DRAM bytes it
    was taken with (bench.py uses the bytes only while the hash matches)."""
    import glob
    import os
    for path in glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")):
        name = os.path.basename(path)[:-3]
        if name.startswith("launches_"):
            continue
        text = open(path, encoding="utf-8").read()
        assert "source_sha256_16:" in text and "dram_bytes_per_launch:" in text, name


def test_committed_profiles_match_the_current_sources():
    """Every committed summary was captured on the kernel sources as they stand:
    a kernel summary's source hash, and each (kernel, hash) pair a launch list
    cites, equal what bench.py computes now, so a kernel change without a new
    capture fails here."""
    import glob
    import os
    import re
    now = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    for path in glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")):
        name = os.path.basename(path)[:-3]
        text = open(path, encoding="utf-8").read()
        if name.startswith("launches_"):
            cited = re.findall(r"(\w+) ([0-9a-f]{16})\b", text)
            assert cited, name
            for kernel, h in cited:
                if kernel in now:
                    assert now[kernel] == h, (name, kernel)
        else:
            kernel = [k for k in now if name.startswith(k)]
            assert len(kernel) == 1, name
            h = re.search(r"source_sha256_16: ([0-9a-f]{16})", text).group(1)
            assert now[kernel[0]] == h, name


def test_oracle_over_all_cores_counts_rows_of_every_process():
    """The all-cores CPU baseline: spawned processes read the batch from shared
    memory, run whole rows and report how many they finished."""
    cfg = W.CONFIGS["tiny"]
    inp = bench.host_inputs(cfg, 0, "steps")
    res = bench.cpu_baseline_all_cores(cfg, inp, budget_s=0.3, path="steps", cores=2)
    assert res["cores"] == 2 and res["kind"] == "oracle" and res["unit"] == "rows/s"
    assert res["value"] > 0 and "processes" in res["sample"]


def test_reference_arm_prints_the_oracle_line(capsys):
    """`bench.py --impl reference`: the oracle over rows on the host cores,
    one JSON line with the reference keys and no GPU."""
    import json
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                       "--warmup", "3"]) == 0
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "rows/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_source_hash_ignores_comments_only(monkeypatch, tmp_path):
    """A profile's hash follows the code: comments may change, code may not."""
    csrc = tmp_path / "dsa_sparse_indexer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "combine.cu").write_text("// a\nint f() { return 1; } /* b */\n")
    h0 = bench.kernel_source_hash("lse_combine")
    (csrc / "combine.cu").write_text("// other words\nint f() { return 1; } /* c\n d */\n")
    assert bench.kernel_source_hash("lse_combine") == h0
    (csrc / "combine.cu").write_text("// a\nint f() { return 2; } /* b */\n")
    assert bench.kernel_source_hash("lse_combine") != h0
