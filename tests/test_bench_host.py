"""Host-side pieces of bench.py that need no GPU: the code hash that keys
recorded DRAM traffic (insensitive to comments and whitespace, sensitive to
code), the traffic lookup, and the decode leg's CPU baseline on a small step
taken from a generator the way the leg takes it."""
import itertools

import numpy as np

import kda_inputs as ki


def _with_source(tmp_path, monkeypatch, text):
    import bench
    d = tmp_path / "kda_linear_attention_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "k.cu").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return bench


def test_code_sha_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    base = "__global__ void k(float *x) {\n    x[0] = 1.f;   // one\n}\n"
    b = _with_source(tmp_path, monkeypatch, base)
    h0 = b.code_sha("k.cu")
    b = _with_source(tmp_path, monkeypatch,
                     "/* header */\n__global__ void k(float *x)\n{\n  x[0] = 1.f; // changed note\n}\n")
    assert b.code_sha("k.cu") == h0
    b = _with_source(tmp_path, monkeypatch, base.replace("1.f", "2.f"))
    assert b.code_sha("k.cu") != h0


def test_traffic_lookup_follows_the_code(tmp_path, monkeypatch):
    import json
    b = _with_source(tmp_path, monkeypatch, "__global__ void k() {}\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = b.code_sha("k.cu")
    (prof / "dram_traffic.json").write_text(json.dumps({"captures": [
        {"kernel": "k_kernel", "code_sha256": sha, "bytes": 12345, "workload": "w"},
        {"kernel": "other", "code_sha256": "0000000000000000", "bytes": 1, "workload": "w"}]}))
    assert b._traffic("k_kernel", "k.cu") == 12345
    assert b._traffic("other", "k.cu") is None          # captured on other code
    assert b._traffic("missing", "k.cu") is None


def test_prefill_traffic_scales_by_units(tmp_path, monkeypatch):
    import json
    b = _with_source(tmp_path, monkeypatch, "__global__ void k() {}\n")
    import os
    os.rename(tmp_path / "kda_linear_attention_gb300" / "csrc" / "k.cu",
              tmp_path / "kda_linear_attention_gb300" / "csrc" / "kda_prefill_split.cu")
    sha = b.code_sha("kda_prefill_split.cu")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.json").write_text(json.dumps({"captures": [
        {"kernel": "intra_chunk_kernel", "code_sha256": sha, "bytes": 1000, "units": 10, "workload": "w"},
        {"kernel": "state_pass_kernel", "code_sha256": sha, "bytes": 500, "units": 10, "workload": "w"}]}))
    t, src = b._prefill_traffic(10)
    assert t == 1500 and "stored" in src
    t, src = b._prefill_traffic(40)
    assert t == 6000 and "scaled" in src


def test_cpu_model_is_a_string():
    import bench
    m = bench.cpu_model()
    assert isinstance(m, str) and m


def test_decode_cpu_baseline_on_a_generated_step():
    import bench
    rng = np.random.Generator(np.random.PCG64(5))
    S0 = ki.gen_decode_state(rng, 3, 2)
    steps = (ki.gen_decode_step(rng, 3, 2, "bf16") for _ in range(4))   # a generator, like the workload's
    steps = iter(steps)
    first = next(steps)
    cpu = bench._decode_cpu_baseline(S0, first, 3, 2)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "GB/s" and cpu["value"] > 0
    assert cpu["cores"] >= 1
    assert sum(1 for _ in itertools.chain([first], steps)) == 4
