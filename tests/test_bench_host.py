"""Host-side bookkeeping of bench.py that needs no GPU: the expert-load
statistics, the output fingerprint and the rerun comparison."""
import hashlib

import pytest

torch = pytest.importorskip("torch")
import bench  # noqa: E402


def test_expert_loads_padding_by_hand():
    # m_e = 0, 1, 128, 129, 300 with 128-row tiles: padded rows 0, 128, 128, 256, 384
    loads = bench.expert_loads(torch.tensor([0, 1, 128, 129, 300]), tile_rows=128)
    A, padded = 558, 896
    assert loads["m_e_max"] == 300 and loads["m_e_min"] == 0
    assert loads["m_e_mean"] == pytest.approx(A / 5)
    assert loads["empty_experts"] == 1
    assert loads["padded_row_frac"] == pytest.approx(round((padded - A) / padded, 4))


def test_expert_loads_whole_tiles_have_no_padding():
    loads = bench.expert_loads([256, 128, 384], tile_rows=128)
    assert loads["padded_row_frac"] == 0.0 and loads["empty_experts"] == 0
    assert bench.expert_loads([0, 0], tile_rows=128)["padded_row_frac"] == 0.0


def test_custom_workload_suffixes_in_any_order():
    s = bench.workload("16384,4096,1536,128,8,1.2,fwd")
    assert (s.N, s.H, s.I, s.E, s.k, s.zipf_s) == (16384, 4096, 1536, 128, 8, 1.2)
    assert not s.backward and s.dtype == "bf16" and s.minibatch_rows == 128
    s = bench.workload("300,512,768,16,4,T=256,fwd,mxfp8")
    assert s.zipf_s is None and s.minibatch_rows == 256 and s.dtype == "mxfp8" and not s.backward
    s = bench.workload("4096,2048,1024,64,8")
    assert s.backward and s.zipf_s is None and s.name == "custom_N4096_H2048_I1024_E64_k8_T128"
    assert bench.workload(None).name.startswith("skewed_fwd_bwd")


def test_digest_is_sha256_of_the_bytes_in_order():
    a = torch.arange(1000, dtype=torch.float32)
    b = torch.arange(77, dtype=torch.int16)
    want = hashlib.sha256(a.numpy().tobytes() + b.numpy().tobytes()).hexdigest()
    # chunk boundaries inside a tensor do not change the digest
    assert bench.output_digest({"a": a, "b": b}, chunk_bytes=96) == want
    assert bench.output_digest({"b": b, "a": a}) != want


def test_rerun_check_sees_a_changed_bit():
    out = {"y": torch.ones(64, dtype=torch.bfloat16), "dx": torch.zeros(8, dtype=torch.float32)}
    same = bench.rerun_check(lambda: None, out)
    assert same["rerun_bitwise_equal"] and same["compared"] == ["y", "dx"]
    assert same["sha256_of"] == ["y", "dx"]

    def flip_sign_of_zero():  # -0.0 == 0.0 as floats, not as bytes
        out["dx"][3] = -0.0
    assert not bench.rerun_check(flip_sign_of_zero, out)["rerun_bitwise_equal"]


def _run_bench(args, env_extra=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, env=env,
                       capture_output=True, text=True, timeout=600, cwd=root)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return r.returncode, [json.loads(ln) for ln in lines]


def test_reference_arm_prints_one_complete_line():
    """The oracle arm's JSON line carries the keys of the bench line, on the
    workload it is given (a tiny one here, so this runs in seconds)."""
    rc, lines = _run_bench(["--impl", "reference", "--config", "256,256,512,8,2",
                            "--steps", "1", "--warmup", "0"])
    assert rc == 0 and len(lines) == 1
    r = lines[0]
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["impl"] == "reference" and r["unit"] == "tokens/s" and r["value"] > 0
    assert r["e2e"]["value"] == r["value"] and r["e2e"]["h2d_bytes_per_step"] == 0
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["cores"] >= 1
    one = r["cpu_baseline"]["one_core"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == "tokens/s"
    assert r["config"]["workload"] == "custom_N256_H256_I512_E8_k2_T128"


def test_reference_arm_on_a_non_zero_rank_exits_quietly():
    rc, lines = _run_bench(["--impl", "reference", "--config", "256,256,512,8,2",
                            "--steps", "1", "--warmup", "0"],
                           {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert rc == 0 and lines == []
