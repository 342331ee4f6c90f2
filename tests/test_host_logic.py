"""Host-side logic that needs no GPU: the layer module's token/head layouts
and GEMM count, and the bench's FLOP split and traffic lookup."""
import os

import torch

import bench
from attention_core_gb300 import layer


def test_layer_layouts_round_trip_and_place_tokens():
    sh = layer.LayerShape(b=2, s=5, h=24, a=3, d=4, ffn=48)
    x = torch.arange(sh.n * sh.a * sh.d, dtype=torch.float32).view(sh.n, sh.a * sh.d)
    heads = layer._heads(x, sh)
    assert heads.shape == (sh.b, sh.a, sh.s, sh.d)
    # token t = batch * s + position, column head * d + c
    for bi, hd, pos, c in ((0, 0, 0, 0), (1, 2, 4, 3), (1, 0, 2, 1)):
        assert heads[bi, hd, pos, c] == x[bi * sh.s + pos, hd * sh.d + c]
    assert torch.equal(layer._tokens(heads, sh), x)


def test_layer_gemm_flops_closed_form():
    sh = layer.LayerShape(b=2, s=2048, h=12288, a=12, d=128, ffn=6144)
    n, h, ad, f = 4096, 12288, 1536, 6144
    assert sh.gemm_flops_fwd() == 2 * n * h * 3 * ad + 2 * n * ad * h + 2 * n * h * f + 2 * n * f * h


def test_layer_weights_are_seeded():
    sh = layer.LayerShape(b=1, s=8, h=16, a=2, d=8, ffn=32)
    w1 = layer.init_weights(sh, seed=3, device="cpu")
    w2 = layer.init_weights(sh, seed=3, device="cpu")
    w3 = layer.init_weights(sh, seed=4, device="cpu")
    assert all(torch.equal(w1[k], w2[k]) for k in w1)
    assert not torch.equal(w1["wqkv"], w3["wqkv"])
    assert w1["wqkv"].dtype == torch.bfloat16 and w1["gamma1"].dtype == torch.float32


def test_bench_kernel_flop_credits_add_up_to_the_method():
    w = dict(b=2, h_q=12, s=2048, d=128)
    fl = bench._flops(w)
    assert fl["k_fwd"] == fl["fwd"]
    assert fl["k_dq"] + fl["k_dkdv"] == fl["bwd"]
    assert fl["fwd"] + fl["bwd"] == fl["total"]
    pairs = 2048 * 2049 // 2
    assert fl["total"] == 14 * 128 * pairs * 2 * 12


def test_traffic_lookup_reads_only_matching_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    cur = bench._csrc_hash()
    (prof / "traffic.txt").write_text("# header\n"
                                      f"attn_fwd_kernel gpt175b 123 {cur}\n"
                                      "attn_bwd_dq_kernel gpt175b 456 000000000000\n")
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_csrc_hash", lambda: cur)
    assert bench._traffic("attn_fwd_kernel", "gpt175b") == 123
    assert bench._traffic("attn_bwd_dq_kernel", "gpt175b") is None      # taken on other sources
    assert bench._traffic("attn_fwd_kernel", "tiny") is None
    assert os.path.isdir(real_root)


def test_source_hash_ignores_comments_only():
    a = "// header\nint f() { return 1; }  // trailing\n/* block\n comment */\nint g;\n"
    b = "int f() { return 1; }\n\nint g;\n"
    c = "int f() { return 2; }\nint g;\n"
    assert bench._strip_comments(a) == bench._strip_comments(b)
    assert bench._strip_comments(a) != bench._strip_comments(c)
