"""Host-side pieces of bench.py that need no GPU: the launch count it
claims for the decode pass and the guard on the committed GEMM traffic
record (taken on the current kernel code, else not reported)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.append(ROOT)

import bench  # noqa: E402


def test_decode_launch_count(monkeypatch):
    # q/k/v in one launch (two Q4_K members and the Q6_K member), o, gate/up
    # in one launch, down: 4 per layer; 5 when the Q6_K member runs alone
    monkeypatch.delenv("RQ_GEMV_NO_DUAL", raising=False)
    assert bench.Stack.decode_launches_per_pass() == 4 * 28
    monkeypatch.setenv("RQ_GEMV_NO_DUAL", "1")
    assert bench.Stack.decode_launches_per_pass() == 5 * 28


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("int f(int x) {  // add one\n  return x + 1;  /* done */\n}\n")
    b.write_text("// a comment\nint f(int x) {\n\n  return x + 1;\n}\n")
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.gemm_code_sha256(str(a)) == bench.gemm_code_sha256(str(b))
    assert bench.gemm_code_sha256(str(a)) != bench.gemm_code_sha256(str(c))


def test_traffic_record_is_guarded(tmp_path, monkeypatch):
    """The committed record parses; with the kernel code changed it is not
    reported (traffic null) instead of being reported stale."""
    rec = os.path.join(ROOT, "profiles", "fp8_gemm_traffic.txt")
    fields = {}
    with open(rec) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    assert int(fields["traffic_bytes_per_launch"]) > 0
    assert len(fields["kernel_code_sha256"]) == 64
    # a copy of the tree whose GEMM code differs reports no traffic
    (tmp_path / "profiles").mkdir()
    with open(rec) as f:
        (tmp_path / "profiles" / "fp8_gemm_traffic.txt").write_text(f.read())
    src = tmp_path / "quantized_linear_layers_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "rq_gemm.cu").write_text("int changed;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.gemm_traffic_per_launch() is None
