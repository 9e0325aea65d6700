"""The committed ncu summaries (CPU only): each names the command that made
it, every ncu command keeps the clocks unlocked (--clock-control none) and
runs committed files only, and each summary whose DRAM traffic the benchmark
reports says which code it was captured on."""
import glob
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))


def test_profiles_are_short_text():
    assert PROFILES
    for p in PROFILES:
        assert p.endswith((".txt", ".md")), p
        assert os.path.getsize(p) < 16 * 1024, p


def test_every_ncu_command_leaves_clocks_alone_and_runs_committed_files():
    for p in PROFILES:
        cmds = [ln.strip() for ln in open(p) if re.match(r"\s*(command:\s*)?ncu\s", ln)]
        assert cmds, f"{p}: no ncu command"
        for c in cmds:
            assert "--clock-control none" in c, f"{p}: {c}"
            assert "_work/" not in c, f"{p}: {c}"
            target = c.split(" python ", 1)[1].split()[0] if " python " in c else None
            assert target is not None and os.path.exists(os.path.join(ROOT, target)), f"{p}: {c}"


def test_traffic_lines_name_their_code():
    for p in PROFILES:
        text = open(p).read()
        if "dram_bytes_per_launch:" in text:
            m = re.search(r"^code_sha256_16:\s*([0-9a-f]{16})", text, flags=re.M)
            assert m, f"{p}: traffic without a code digest"


def test_current_attention_profiles_feed_the_bench():
    """The attention summaries were taken on the current kernel source, so the
    bench line carries their DRAM traffic.  After a change to the attention
    code, recapture them (the commands are in the files) before committing."""
    src = os.path.join(ROOT, "offloaded_kv_decode_gb300", "csrc", "clo_attention.cu")
    for wl in ("llama3_8b_layer_b8_32k", "llama3_8b_step_b1_128k", "llama3_8b_step_b4_128k",
               "qwen25_14b_step_b16_64k", "paged_llama2_7b_b256"):
        assert bench.traffic_from_profiles(src, "attn_split_kernel", wl) is not None, wl
