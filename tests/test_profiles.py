"""The committed ncu summaries under profiles/: text only, each with the commands that made
it, every ncu command leaving the GPU clocks alone, and every counter record pointing at a
summary that exists. (No GPU needed.)"""
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def test_profiles_hold_text_summaries_only():
    for f in os.listdir(PROFILES):
        assert os.path.splitext(f)[1] in (".md", ".txt", ".json"), f"{f}: raw captures stay out of profiles/"
        assert os.path.getsize(os.path.join(PROFILES, f)) < 64 * 1024, f"{f}: a summary is a few KB"


def test_every_summary_gives_its_commands_and_ncu_never_locks_clocks():
    for f in _summaries():
        text = open(os.path.join(PROFILES, f), encoding="utf-8").read()
        text = re.sub(r"\\\n\s*", " ", text)               # join backslash-continued lines
        commands = [ln.strip() for ln in text.splitlines() if re.match(r"\s*ncu\s+-", ln)]
        assert commands, f"{f}: no ncu command line"
        for c in commands:
            assert "--clock-control none" in c, f"{f}: {c[:80]}"


def test_counter_records_point_at_existing_summaries():
    with open(os.path.join(PROFILES, "ncu_traffic.json")) as fh:
        recs = json.load(fh)
    for name, rec in recs.items():
        if not isinstance(rec, dict) or "source" not in rec:
            continue
        assert os.path.exists(os.path.join(ROOT, rec["source"])), f"{name}: {rec['source']}"
        assert re.fullmatch(r"[0-9a-f]{16}", rec["kernel_sha"]), name
