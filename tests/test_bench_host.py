"""The bench's host-side bookkeeping on the CPU: the source hash that decides
whether the recorded DRAM traffic still describes the kernels."""
import os

import bench


def test_code_only_drops_comments_and_layout():
    src = "int a = 1;  // one\n/* block\n comment */ int  b =\n 2; // two\n"
    assert bench._code_only(src) == "int a = 1; int b = 2;"


def _hash_of(tmp_path, monkeypatch, text):
    csrc = tmp_path / "hyper_connection_residual_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cuh").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return bench.kernel_source_hash(("k.cuh",))


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    base = _hash_of(tmp_path, monkeypatch, "__global__ void k() { x = 1; }\n")
    commented = _hash_of(tmp_path, monkeypatch, "// the kernel\n__global__ void k() {\n  x = 1;  /* set */\n}\n")
    changed = _hash_of(tmp_path, monkeypatch, "__global__ void k() { x = 2; }\n")
    assert commented == base
    assert changed != base


def test_recorded_traffic_is_read_only_for_matching_sources(tmp_path, monkeypatch):
    # profiles/traffic.json is read from the repository; with the sources
    # pointed elsewhere the hash no longer matches and no traffic is reported.
    real_root = bench.ROOT
    assert os.path.exists(os.path.join(real_root, "profiles", "traffic.json"))
    csrc = tmp_path / "hyper_connection_residual_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.T1_KERNEL_SOURCES:
        (csrc / name).write_text("// nothing\n")
    (tmp_path / "profiles").mkdir()
    with open(os.path.join(real_root, "profiles", "traffic.json")) as f:
        (tmp_path / "profiles" / "traffic.json").write_text(f.read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic() is None
