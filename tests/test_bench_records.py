"""bench.py's link between recorded ncu counters and the kernel sources: the key is a hash of the
sources' code, so an edit of a comment or of whitespace keeps the recorded traffic while any change
of code retires it; and the committed traffic lines resolve for the sources as they stand."""
import os
import shutil

import pytest


def _copy_tree(tmp_path):
    import bench
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "moe_expert_layer_routing_gb300", "csrc"),
                    root / "moe_expert_layer_routing_gb300" / "csrc",
                    ignore=shutil.ignore_patterns("_build", "*.o"))
    return root


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    import bench
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.source_sha()
    f = root / "moe_expert_layer_routing_gb300" / "csrc" / "reduce.cu"
    text = f.read_text()
    f.write_text("// a new line comment\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3))
    assert bench.source_sha() == base
    f.write_text(text.replace("acc[2 * j] +=", "acc[2 * j] -=", 1))
    assert bench.source_sha() != base


def test_committed_traffic_lines_match_the_sources():
    import bench
    sha = bench.source_sha()
    path = os.path.join(bench.ROOT, "profiles", "gemm_traffic_imbalanced_mxfp8.md")
    if sha not in open(path).read():
        pytest.skip("kernel code changed since the traffic capture (bench then reports traffic null)")
    for stage in ("G1_dA_dswiglu", "G3_dW2", "G2_dx_expanded", "G4_dW1"):
        assert bench.recorded_traffic("imbalanced_mxfp8", stage) > 0
