"""Host logic of bench.py that needs no GPU: the DRAM-traffic record is used
only while the kernel's source files are the ones it was captured on
(comments and whitespace aside), and the roofline helpers."""
import json
import os
import shutil

import bench


def _copy_tree(tmp_path):
    """A copy of the kernel sources and the traffic record under tmp_path."""
    src = os.path.join(bench.ROOT, "int4_gathered_expert_gb300", "csrc")
    dst = tmp_path / "int4_gathered_expert_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in set(sum(bench.KERNEL_SOURCES.values(), ())):
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"), tmp_path / "profiles" / "traffic.json")
    return dst


def test_digest_ignores_comments_and_whitespace_but_not_code(tmp_path, monkeypatch):
    dst = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    kernel = "k_umma2<1>"
    f = dst / "e0_prefill.cu"
    base = bench.kernel_source_digest(kernel)
    decode = bench.kernel_source_digest("k_stack_ll")
    text = f.read_text(encoding="utf-8")
    f.write_text("// a new comment line\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3),
                 encoding="utf-8")
    assert bench.kernel_source_digest(kernel) == base
    f.write_text(text.replace("constexpr int STAGES = 4;", "constexpr int STAGES = 3;"), encoding="utf-8")
    assert bench.kernel_source_digest(kernel) != base
    # the decode kernel does not read this file
    assert bench.kernel_source_digest("k_stack_ll") == decode


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    dst = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = json.loads((tmp_path / "profiles" / "traffic.json").read_text())
    for kernel, entry in rec.items():
        assert kernel in bench.KERNEL_SOURCES
        assert entry["dram_bytes_per_launch"] == entry["read_bytes"] + entry["write_bytes"]
        # a record taken on these sources is used
        entry["source_digest"] = bench.kernel_source_digest(kernel)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    for kernel, entry in rec.items():
        assert bench.recorded_traffic(kernel) == entry["dram_bytes_per_launch"]
    # a code change in one kernel's sources voids that kernel's record only
    f = dst / "e0_stack_ll.cuh"
    f.write_text(f.read_text(encoding="utf-8") + "\nconstexpr int LL_UNUSED = 1;\n", encoding="utf-8")
    assert bench.recorded_traffic("k_stack_ll") is None
    assert bench.recorded_traffic("k_umma2<1>") == rec["k_umma2<1>"]["dram_bytes_per_launch"]
    assert bench.recorded_traffic("no_such_kernel") is None


def test_algorithmic_bytes_of_a_35b_token():
    """The roofline's numerator for the 35B stack, spelled out: an expert is
    3 H I / 2 code bytes plus 4 bytes (fp16 scale and bias) per 64-group,
    2 I H / 64 + H I / 64 groups; 40 layers, K = 4, a shared expert with a
    rank-16 LoRA on gate, up and down, 33 heads of hidden 512 (fc1 and Lres
    over h plus their 2K one-hot columns, fc2, b1, b2), 7 native routers."""
    from int4_gathered_expert_gb300 import synth
    H, I, E, K, L, r, hid = 2048, 512, 256, 4, 40, 16, 512
    expert = 3 * H * I // 2 + 4 * (2 * I * H // 64 + H * I // 64)
    assert expert == 1_769_472
    nb = bench.bytes_per_token(synth.STACK35B, native_layers=7)
    assert nb["routed"] == L * K * expert == 283_115_520
    assert nb["shared"] == L * expert
    assert nb["lora"] == L * 2 * r * (2 * (H + I) + (I + H)) == 9_830_400
    head = hid * H * 2 + E * H * 2 + E * hid * 2 + 2 * K * (hid + E) * 2 + (hid + E) * 2
    assert nb["heads"] == 33 * head == 112_915_968
    assert nb["routers"] == 7 * E * H * 2
    assert nb["total"] == sum(nb[k] for k in ("routed", "shared", "lora", "heads", "routers"))
    assert abs(nb["total"] / 1e6 - 484.0) < 0.1


def test_whole_job_rate():
    assert bench.whole_job_rate(256, 4, 2.0) == 512.0
    assert bench.whole_job_rate(256, 1, 0.5) == 512.0
