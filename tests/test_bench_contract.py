"""Host-side checks of the benchmark: the roofline's algorithmic bytes equal
the bytes of the tensors a step reads (counted from the generated weights,
not from the formula), and the reference arm prints one JSON line with the
contract's keys. CPU only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decode_megakernel_llama_gb300 import synth  # noqa: E402
from decode_megakernel_llama_gb300.configs import LLAMA_1B, TINY, ModelShape  # noqa: E402


@pytest.mark.parametrize("shape", [TINY, ModelShape("odd", 3, 768, 12, 4, 64, 3072, 1000, 1e-5, 1e4)])
def test_algorithmic_bytes_match_the_generated_tensors(shape):
    w = synth.make_weights(shape, "cpu", 0)
    tensors = [w["embed"], w["final_norm"]] + [t for lw in w["layers"] for t in lw.values()]
    weight_bytes = sum(t.numel() * t.element_size() for t in tensors)
    row = shape.d_model * 2  # the embedding row gathered for the token, besides the LM head's full read
    for pos in (0, 5, 37):
        kv = 2 * shape.n_layers * shape.n_kv_heads * (pos + 1) * shape.head_dim * 2  # K and V, bf16
        assert bench.algorithmic_bytes(shape, pos) == weight_bytes + row + kv


def test_llama1b_bytes_per_step():
    # 1.2358 G bf16 weights (embedding counted for the LM head and once more
    # for the gathered row) + 32 KB of keys/values per attended position
    assert bench.algorithmic_bytes(LLAMA_1B, 0) == 2_471_632_896 + 32_768


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["steps"] == 2 and line["warmup"] == 1 and line["higher_is_better"] is False
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "tiny shape" in line["config"]["workload"]
    # the same positions the GPU arm times: after the 8-token prompt
    assert "timed decode positions 8..9" in line["config"]["workload"]
    assert cb["cpu_model"] and cb["affinity_cores"] >= 1


def test_cpu_baseline_reports_all_cores_and_one_thread():
    w = synth.host_weights(synth.make_weights(TINY, "cpu", 0))
    prompt = synth.prompt_tokens(TINY.vocab, 8)
    cb = bench.oracle_baseline(TINY, w, prompt, 8, 3, 0.5, 0.5)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert "positions 8.." in cb["sample"] and cb["cpu_model"]


def test_kernel_hash_covers_every_source_of_the_megakernel():
    # the committed DRAM-traffic record is matched to the kernel by this hash,
    # so every file that shapes the megakernel's code or plan must be in it
    # (the allocation-free entry point's unit only moves its scratch; the
    # W2A8 GEMV's, the prefill's and the sparse FFN's units are separate kernels)
    from decode_megakernel_llama_gb300 import build as mkbuild
    import inspect
    src = inspect.getsource(bench.kernel_sha)
    for f in mkbuild.DEPS:
        if f in ("mk_noalloc.cu", "mk_internal.h", "mk_w2a8.cu", "mk_prefill.cu", "mk_prefill.h", "mk_twell.cu"):
            continue
        assert f'"{f}"' in src, f
