"""Host-side arithmetic of bench.py (no GPU): the roofline's algorithmic bytes and FLOPs for the
dense batch, and the rule that ties the recorded DRAM traffic to the kernel sources it was
measured on."""
import json
import os

import bench


def test_algorithmic_bytes_dense_batch():
    """The forward's minimum traffic on the dense batch (8 x 8192 tokens, 32 heads, K = V = 128,
    fp32 start state, final state and checkpoint rows every 1024 tokens), summed tensor by
    tensor from the shapes."""
    T, N, H, K, V = 65536, 8, 32, 128, 128
    rows = N * (8192 // 1024)  # one checkpoint row per 1024 tokens of each sequence, entry 0 included
    q = k = T * H * K * 2
    v = o = T * H * V * 2
    g = beta = T * H * 4
    s0 = final = N * H * K * V * 4
    ckpt = rows * H * K * V * 4
    cu = (N + 1) * 4
    want = q + k + v + o + g + beta + s0 + final + ckpt + cu
    assert want == 2_332_033_060
    assert bench.algorithmic_bytes(T, N, H, H, K, V, rows) == want
    # no start state, no final state, bf16 rows: each term leaves on its own
    assert bench.algorithmic_bytes(T, N, H, H, K, V, rows, s0=False, final=False, ckpt_bytes=2) == \
        want - s0 - final - ckpt // 2


def test_algorithmic_flops_per_chunk_head():
    """Per 64-token chunk and head with d = 128: five C x C x d products (K K^T, Q K^T, T (beta V),
    T (beta gamma K), the intra-chunk output) and three C x d x d (W S, Q S, the state update),
    2 flops per multiply-add; a ragged last chunk counts whole."""
    C, d = 64, 128
    per = 5 * 2 * C * C * d + 3 * 2 * C * d * d
    assert per == 11_534_336
    assert bench.algorithmic_flops([8192] * 8, 32, d, d) == 8 * 128 * 32 * per
    assert bench.algorithmic_flops([1, 64, 65], 1, d, d) == (1 + 1 + 2) * per
    assert bench.algorithmic_flops([0], 4, d, d) == 0


def test_code_only_ignores_comments_and_blank_lines():
    src = "int a = 1;  // one\n\n/* block\n   comment */\nint b = a + 1;\n"
    same = "int a = 1;\n// a note\nint b = a + 1;  /* two */\n\n"
    other = "int a = 1;\nint b = a + 2;\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)


def _fake_tree(root, code):
    csrc = os.path.join(root, "gated_delta_rule_29_gb300", "csrc")
    os.makedirs(csrc)
    for name in bench.TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name), "w") as f:
            f.write(code + "// " + name + "\n")
    os.makedirs(os.path.join(root, "profiles"))


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The traffic recorded with a hash of the kernel sources is reported while those sources
    are unchanged (comments aside) and withheld (None) once their code differs."""
    root = str(tmp_path)
    _fake_tree(root, "int x = 1;\n")
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.profiled_traffic() is None  # no record yet
    rec = {"kernel_source_hash": bench.kernel_source_hash(), "traffic_bytes_per_launch": 123.0}
    with open(os.path.join(root, "profiles", "gdn_fwd_two_pass_dense_batch.json"), "w") as f:
        json.dump(rec, f)
    assert bench.profiled_traffic() == 123.0
    chunk = os.path.join(root, "gated_delta_rule_29_gb300", "csrc", "gdn_chunk.cu")
    with open(chunk, "a") as f:
        f.write("// a comment changes nothing\n")
    assert bench.profiled_traffic() == 123.0
    with open(chunk, "a") as f:
        f.write("int y = 2;\n")
    assert bench.profiled_traffic() is None


def test_committed_traffic_record_names_its_sources():
    """The committed record covers both forward passes and the sources the hash is taken over."""
    with open(os.path.join(bench.ROOT, "profiles", "gdn_fwd_two_pass_dense_batch.json")) as f:
        rec = json.load(f)
    assert tuple(rec["hashed_sources"]) == bench.TRAFFIC_SOURCES
    parts = sum(rec["dram_bytes_read"].values()) + sum(rec["dram_bytes_write"].values())
    assert rec["traffic_bytes_per_launch"] == parts
