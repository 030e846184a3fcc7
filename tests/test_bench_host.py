"""Host-side bookkeeping of bench.py (CPU): the source hash that ties the
committed ncu traffic figures to the kernel code, and the lookup of those
figures."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_code_only_drops_comments_keeps_literals():
    src = 'int a = 1;  // trailing\n/* block\n comment */ const char* s = "//x /*y*/";\nchar q = \'"\';'
    assert bench._code_only(src) == 'int a = 1; const char* s = "//x /*y*/"; char q = \'"\';'


def test_code_only_ignores_layout_not_code():
    a = "int f(int x) {\n    return x + 1;  // one\n}\n"
    b = "int f(int x) { return x + 1; }"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """A summary taken on the current code gives its traffic; one taken on
    other code (another hash) gives none."""
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda: "0123456789abcdef")
    f = tmp_path / "profiles" / "moe_megakernel_mixtral.md"
    f.write_text("source_hash: 0123456789abcdef\ntraffic_bytes_per_launch: 2334009830\n")
    assert bench.profiled_traffic("mixtral") == 2334009830.0
    f.write_text("source_hash: fedcba9876543210\ntraffic_bytes_per_launch: 2334009830\n")
    assert bench.profiled_traffic("mixtral") is None
    assert bench.profiled_traffic("fine") is None  # no summary at all


def test_default_line_carries_the_secondary_sweeps(monkeypatch):
    """The default run adds the other configurations' records (fine-grained
    layer, fused Mixtral-shaped block, split-K GEMM, MLP chain, warm-up) to
    its line; here each measurement is a fake that checks what it is given."""
    import argparse

    import torch

    seen = []

    def fake_moe(cfg, Fs, device, steps, warmup):
        assert Fs is None or isinstance(Fs, int)
        assert isinstance(device, torch.device)
        seen.append((cfg.name, Fs, steps, warmup))
        return {"value": 1.0}

    def fake_dense(kind, device, steps, warmup):
        assert kind in ("splitk", "mlp") and isinstance(device, torch.device)
        seen.append((kind, steps, warmup))
        return {"sweep": []}

    monkeypatch.setattr(bench, "moe_sweep_record", fake_moe)
    monkeypatch.setattr(bench, "dense_sweep_record", fake_dense)
    monkeypatch.setattr(bench, "run_warmup", lambda args: {"value": 2.0})
    args = argparse.Namespace(steps=7, warmup=3, no_warmup_record=False)
    out = bench.secondary_sweeps(args, torch.device("cpu"))
    assert set(out) == {"fine", "mixtral_block", "splitk", "mlp", "warmup"}
    assert ("fine_skewed", None, 7, 3) in seen and ("mixtral", 0, 7, 3) in seen
    assert ("splitk", 7, 3) in seen and ("mlp", 7, 3) in seen
    assert out["warmup"] == {"value": 2.0}
