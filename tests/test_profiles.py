"""The committed profile summaries: every ncu command they record leaves the
GPU clocks alone and runs only committed files, and every per-launch DRAM
record names a source and a summary that exist.  CPU only."""
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROF = os.path.join(ROOT, "profiles")


def _commands(text):
    """Shell commands in the fenced blocks, backslash continuations joined."""
    cmds = []
    for block in re.findall(r"```[a-z]*\n(.*?)```", text, re.S):
        cur = ""
        for line in block.splitlines():
            cur += line.rstrip()
            if cur.endswith("\\"):
                cur = cur[:-1] + " "
                continue
            if cur.strip():
                cmds.append(cur.strip())
            cur = ""
        if cur.strip():
            cmds.append(cur.strip())
    return cmds


def _summaries():
    return sorted(f for f in os.listdir(PROF) if f.endswith(".md") and f != "README.md")


def test_every_summary_records_a_command():
    for f in _summaries():
        cmds = _commands(open(os.path.join(PROF, f)).read())
        assert any(c.startswith(("ncu ", "python ")) for c in cmds), f


def test_ncu_commands_keep_the_clocks():
    n = 0
    for f in _summaries():
        for c in _commands(open(os.path.join(PROF, f)).read()):
            if c.startswith("ncu "):
                n += 1
                assert "--clock-control none" in c, (f, c)
    assert n > 0


def test_commands_run_committed_files_only():
    for f in _summaries():
        for c in _commands(open(os.path.join(PROF, f)).read()):
            assert "_work" not in c, (f, c)
            for script in re.findall(r"python\s+(\S+\.py)", c):
                assert os.path.exists(os.path.join(ROOT, script)), (f, script)


def test_traffic_records_name_existing_sources_and_summaries():
    recs = json.load(open(os.path.join(PROF, "traffic.json")))
    assert recs
    for key, r in recs.items():
        assert os.path.exists(os.path.join(ROOT, r["source"])), key
        assert os.path.exists(os.path.join(ROOT, r["capture"])), key
        assert re.fullmatch(r"[0-9a-f]{16}", r["source_sha256_16"]), key
        assert r["dram_bytes_per_launch"] > 0, key
        assert "--clock-control none" in r.get("capture_command", "--clock-control none"), key


def test_index_lists_every_summary():
    index = open(os.path.join(PROF, "README.md")).read()
    for f in _summaries():
        assert f"`{f}`" in index, f


def test_traffic_of_the_bench_line_kernels_is_current():
    """The bench line reports `roofline.traffic` only for kernel source the
    DRAM counters were taken on.  The committed records of the kernels the
    line names are current, and a record whose source changed reads as None."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for key in ("gemv_gateup", "gemm_tc_gateup_b32", "decode_persistent_b1"):
        assert bench.traffic_record(key) is not None, key
    assert bench.traffic_record("no_such_kernel") is None


def test_stale_traffic_record_reads_as_none(tmp_path, monkeypatch):
    import shutil
    import sys
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    rec = json.load(open(os.path.join(PROF, "traffic.json")))["gemv_gateup"]
    src = tmp_path / rec["source"]
    src.parent.mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, rec["source"]), src)
    json.dump({"gemv_gateup": rec}, open(tmp_path / "profiles" / "traffic.json", "w"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("gemv_gateup") == rec["dram_bytes_per_launch"]
    with open(src, "a") as f:
        f.write("\n// edited\n")
    assert bench.traffic_record("gemv_gateup") is None
