"""Host-side pieces of bench.py that its JSON line depends on (no GPU):
the hash that ties recorded ncu traffic to the library's code, and the
lookup of that traffic."""
import json
import os

import bench


def test_code_hash_ignores_comments_and_layout():
    src = "int f(int a) {\n    // doubled\n    return 2 * a; /* fast */\n}\n"
    same = "int f(int a) { return 2 * a; }  // reformatted, comment moved\n"
    other = "int f(int a) {\n    return 3 * a;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    multi = "/* a\n multi-line\n comment */ int x;"
    assert bench._code_only(multi) == "int x;"


def test_recorded_traffic_is_tied_to_the_code(tmp_path, monkeypatch):
    sha = bench.kernel_sha()
    assert len(sha) == 16
    # a copy of the tree with the real sources and a traffic record of its own
    pkg = tmp_path / "decode_megakernel_persistent_gb300"
    pkg.mkdir()
    os.symlink(os.path.join(bench.ROOT, "decode_megakernel_persistent_gb300", "csrc"), pkg / "csrc")
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"megakernel:w": {"kernel_sha": sha, "bytes_per_launch": 123},
           "megakernel:old": {"kernel_sha": "0" * 16, "bytes_per_launch": 456}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_sha() == sha
    assert bench.recorded_traffic("w", "megakernel") == 123
    assert bench.recorded_traffic("old", "megakernel") is None  # taken on other code
    assert bench.recorded_traffic("missing", "megakernel") is None
    assert bench.recorded_traffic("w", "chain") is None


def test_kernel_sha_covers_the_backends_own_sources(tmp_path, monkeypatch):
    # a tree of stand-in sources: the megakernel's hash moves with the megakernel's
    # files and the shared runtime, not with the prefill or chain files
    csrc = tmp_path / "decode_megakernel_persistent_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("megakernel.cuh", "chain.cu", "prefill.cu", "api.cpp"):
        (csrc / name).write_text(f"int {name.split('.')[0]};")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    mk, ch = bench.kernel_sha("megakernel"), bench.kernel_sha("chain")
    (csrc / "prefill.cu").write_text("int changed;")
    assert (bench.kernel_sha("megakernel"), bench.kernel_sha("chain")) == (mk, ch)
    (csrc / "chain.cu").write_text("int changed;")
    assert bench.kernel_sha("megakernel") == mk and bench.kernel_sha("chain") != ch
    ch = bench.kernel_sha("chain")
    (csrc / "megakernel.cuh").write_text("int changed;")
    assert bench.kernel_sha("megakernel") != mk and bench.kernel_sha("chain") == ch
    mk = bench.kernel_sha("megakernel")
    (csrc / "api.cpp").write_text("int changed;")
    assert bench.kernel_sha("megakernel") != mk and bench.kernel_sha("chain") != ch


def test_clock_summary_reads_samples_inside_the_timed_region(monkeypatch):
    # no nvidia-smi here: the sampler still records marks and parses what its
    # output file holds; samples outside the marks are ignored, "Not Active"
    # is not a throttle reason
    import subprocess
    import time as _time

    def no_smi(*a, **k):
        raise OSError("no nvidia-smi")

    monkeypatch.setattr(subprocess, "Popen", no_smi)
    cs = bench.ClockSampler(0)
    assert cs.proc is None
    t0 = _time.time()
    cs.marks = [t0, t0 + 10.0]

    def stamp(t):
        lt = _time.localtime(t)
        return _time.strftime("%Y/%m/%d %H:%M:%S", lt) + ".500"

    rows = [
        (t0 - 60, 900, "Active", "Not Active"),      # before the timed region: ignored
        (t0 + 1, 2070, "Not Active", "Not Active"),
        (t0 + 2, 2070, "Not Active", "Active"),      # power cap during the region
        (t0 + 3, 2055, "Not Active", "Not Active"),
        (t0 + 60, 500, "Active", "Not Active"),      # after: ignored
    ]
    with open(cs.out.name, "w") as f:
        for t, mhz, hw, cap in rows:
            f.write(f"{stamp(t)}, 0, {mhz}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, {cap}\n")
    cs.stop()
    r = cs.summary()
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2070
    assert r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_prefill_tensor_flops_count_each_gemms_terms():
    from decode_megakernel_persistent_gb300 import synth
    H, q, kv, I, L, n = 2048, 2048, 512, 8192, 16, 1024
    want = 2.0 * n * L * (3 * (q * H + 2 * kv * H) + 2 * (H * q + 2 * I * H + H * I))
    assert bench.prefill_tensor_flops(synth.LLAMA_1B, n) == want
