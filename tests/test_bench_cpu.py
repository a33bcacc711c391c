"""The benchmark's host-side paths that need no GPU: the reference arm (the
CPU oracle on bounded samples) as a single process and as a two-rank
torchrun job over gloo, where rank 0 alone prints the JSON line."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_line(line, n):
    assert line["impl"] == "reference"
    assert line["n_gpus"] == n and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "decode-L1"


def test_reference_arm_single_process():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
           "--workload", "decode-L1", "--shrink", "64"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1)


def test_reference_arm_two_ranks_gloo():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "decode-L1", "--shrink", "64"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2)


def test_kernel_names_mirror_the_dispatch():
    """The bench names the kernels the library dispatches: the tcgen05 prefill
    for every rule at dk = dv = 128 with fp16 activations (per-key decay and
    GDN-2 through the per-key prepare pass when their gates are fp32), the
    warp-level MMA kernel for other shapes, the token-serial kernels otherwise."""
    import importlib.util
    sys.path.insert(0, ROOT)
    import workloads
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    base = dict(seed=1, B=1, lengths=[8], hq=1, hv=1, dk=128, dv=128, act="f16")
    cases = [
        (dict(rule="gated_delta"), "chunk_prepare_kernel<1>+chunk_chain_kernel<2>"),
        (dict(rule="linear"), "chunk_prepare_kernel<0>+chunk_chain_kernel<0>"),
        (dict(rule="gated"), "chunk_prepare_kernel<0>+chunk_chain_kernel<1>"),
        (dict(rule="gdn2", decay_per_key=True, gate_dtype="f32"),
         "chunk_prepare_perkey_kernel<1>+chunk_chain_kernel<2>"),
        (dict(rule="gated_delta", decay_per_key=True, gate_dtype="f32"),
         "chunk_prepare_perkey_kernel<0>+chunk_chain_kernel<2>"),
        (dict(rule="gated_delta", decay_per_key=True, lengths=[200]),
         "chunk_prepare_perkey_kernel<0>+chunk_chain_kernel<2>"),
        (dict(rule="gated_delta", decay_per_key=True, lengths=[200], dk=64, dv=64), "recurrent_long_kernel<64>"),
        (dict(rule="gated", decay_per_key=True, gate_dtype="f32"),
         "chunk_prepare_perkey_kernel<0>+chunk_chain_kernel<2>"),
        (dict(rule="gated", decay_per_key=True), "chunk_prepare_perkey_kernel<0>+chunk_chain_kernel<2>"),
        (dict(rule="gated", decay_per_key=True, dk=64, dv=64), "recurrent_pipe_kernel<64,false>"),
        (dict(rule="gdn2", decay_per_key=True, gate_dtype="f32", erase="input", write_gate="input"),
         "chunk_prepare_perkey_kernel<1>+chunk_chain_kernel<2>"),
        (dict(rule="gated_delta", dk=64, dv=64), "chunked_mma_kernel<64,false>"),
    ]
    for over, name in cases:
        kw = dict(base)
        kw.update(over)
        p = workloads.make(**kw)
        assert b.kernel_name(p, "chunked") == name, (over, b.kernel_name(p, "chunked"))
        gate16 = over.get("decay_per_key") and "gate_dtype" not in over and "chain" in name
        assert b.launches_per_call(p, "chunked") == ((4 if gate16 else 3) if "chain" in name else 1)
    p = workloads.make(**dict(base, rule="gated_delta", act="f32"))
    assert b.kernel_name(p, "chunked") == "chunk_prepare_kernel<1>+chunk_chain_kernel<2>"
    assert b.launches_per_call(p, "chunked") == 6
    p = workloads.decode(1, B=4, num_slots=8)
    assert b.kernel_name(p, "recurrent") == "recurrent_pipe_kernel<128,false>"
    p = dict(p, state_kmajor=True)
    assert b.kernel_name(p, "recurrent") == "recurrent_pipe_kernel<128,true>"
