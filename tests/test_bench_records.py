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


@pytest.mark.parametrize("name", ["tiny_bf16", "dense_mxfp8_4096", "bias_bf16", "small_mxfp8"])
def test_resident_input_bytes_match_the_tensors(name):
    """The L2 statement of the JSON line rests on the resident input bytes, computed from the shapes: they
    equal the bytes of the tensors a step holds (MXFP8 weights as codes and one scale byte per 32)."""
    import bench
    from moe_expert_layer_routing_gb300.inputs import (CONFIGS, LinearConfig, make_linear_inputs, make_moe_inputs,
                                                       small_moe)
    cfg = {"bias_bf16": small_moe("b", T=300, H=256, I=256, E=8, K=3, B=256, bias=True),
           "small_mxfp8": small_moe("m", T=300, H=256, I=256, E=8, K=3, B=256, precision=1)}.get(name) or CONFIGS[name]
    if isinstance(cfg, LinearConfig):
        inp = make_linear_inputs(cfg)
        held = sum(t.numel() * t.element_size() for t in (inp.dY, inp.W, inp.X))
    else:
        inp = make_moe_inputs(cfg)
        held = sum(t.numel() * t.element_size() for t in [inp.x, inp.dout, inp.s, inp.ids, inp.ckpt] +
                   ([inp.b2] if cfg.bias else []))
        w = inp.W1.numel() + inp.W2.numel()
        held += w + w // 32 if cfg.precision == 1 else 2 * w
    assert bench.resident_input_bytes(cfg) == held
    l2 = 132 * 2 ** 20
    note = bench.l2_note(held, l2)
    assert note.startswith("L2 flushed" if held <= l2 else "inputs larger than L2")
