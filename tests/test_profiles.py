"""The committed ncu summaries under profiles/ stay what they claim to be: each
gives the full command that produced it, with --clock-control none, running
committed files only; the traffic records name sources that exist; nothing
under profiles/ is a raw report or runnable."""
import json
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROF = os.path.join(ROOT, "profiles")


def _tracked():
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    return set(out.stdout.split()) if out.returncode == 0 else None


def test_every_summary_gives_its_ncu_command():
    mds = [f for f in os.listdir(PROF) if f.endswith(".md")]
    assert mds
    tracked = _tracked()
    for f in mds:
        text = open(os.path.join(PROF, f)).read()
        cmds = [ln.strip() for ln in text.splitlines() if ln.strip().startswith("ncu ")]
        assert cmds, f"{f}: no ncu command"
        for c in cmds:
            assert "--clock-control none" in c, f"{f}: {c}"
            m = re.search(r"python (\S+\.py)", c)
            assert m, f"{f}: the command runs no script"
            assert os.path.exists(os.path.join(ROOT, m.group(1))), f"{f}: {m.group(1)}"
            if tracked is not None:
                assert m.group(1) in tracked, f"{f}: {m.group(1)} is not committed"


def test_traffic_records_name_existing_sources():
    with open(os.path.join(PROF, "traffic.json")) as fh:
        d = json.load(fh)
    for key, e in d.items():
        src = os.path.join(ROOT, "quantized_decode_attention_blocks_b300", "csrc", e["source"])
        assert os.path.exists(src), key
        assert e["dram_bytes_per_launch"] > 0 and len(e["source_sha256_16"]) == 16
        assert "--clock-control none" in e["capture"]


def test_profiles_hold_text_only():
    for f in os.listdir(PROF):
        assert os.path.splitext(f)[1] in (".md", ".txt", ".json"), f
