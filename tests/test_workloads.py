"""The seeded input recipe: deterministic by seed, and each ingredient (sink
prefix, needle blocks, skip-tier key scale, bf16 rounding of an fp32 draw)
present with the properties the recipe states.  CPU only."""
import math

import torch

from block_sparse_gated_gb300 import workloads as wl


def test_same_seed_same_tensors_and_different_seed_different_tensors():
    a = wl.layer_inputs(4, 2, 300, 64, 5, needles=2, sink_tokens=16, skip_rate=0.3, block=64)
    b = wl.layer_inputs(4, 2, 300, 64, 5, needles=2, sink_tokens=16, skip_rate=0.3, block=64)
    c = wl.layer_inputs(4, 2, 300, 64, 6, needles=2, sink_tokens=16, skip_rate=0.3, block=64)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x, y)
    assert a.needle_blocks == b.needle_blocks
    assert torch.equal(a.skip_tier, b.skip_tier)
    assert not torch.equal(a.q, c.q)


def test_bf16_and_fp16_come_from_the_same_fp32_draw():
    x = wl.layer_inputs(2, 1, 256, 64, 9)
    y = wl.layer_inputs(2, 1, 256, 64, 9, dtype=torch.float16)
    assert x.q.dtype == torch.bfloat16 and y.q.dtype == torch.float16
    fp32 = wl.gaussian((2, 256, 64), 9, 0)
    assert torch.equal(x.q, fp32.to(torch.bfloat16))
    assert torch.equal(y.q, fp32.to(torch.float16))


def test_sink_prefix_scales_the_first_keys():
    plain = wl.layer_inputs(2, 2, 512, 128, 11)
    sink = wl.layer_inputs(2, 2, 512, 128, 11, sink_tokens=256, sink_scale=4.0)
    ratio = sink.k[:, :256].float().norm() / plain.k[:, :256].float().norm()
    assert abs(float(ratio) - 4.0) < 0.05
    assert torch.equal(sink.k[:, 256:], plain.k[:, 256:])


def test_needle_blocks_point_along_the_mean_query_direction():
    Hq, Hkv, L, d, B = 4, 2, 2048, 128, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 13, needles=3, sink_tokens=256, block=B)
    g = Hq // Hkv
    qf = x.q.float().view(Hkv, g, L, d).mean(dim=(1, 2))
    u = qf / qf.norm(dim=-1, keepdim=True)
    for kh, blocks in enumerate(x.needle_blocks):
        assert len(blocks) == 3 and len(set(blocks)) == 3
        assert all(j * B >= 256 for j in blocks)  # past the sink prefix
        proj = (x.k[kh].float() @ u[kh]).view(-1, B).mean(dim=1)  # mean projection per block
        for j in range(L // B):
            if j in blocks:
                assert proj[j] > 0.5 * 4.0 * math.sqrt(d)
            else:
                assert abs(float(proj[j])) < 1.0


def test_skip_tier_scales_whole_key_blocks_and_spares_block_zero():
    x = wl.layer_inputs(2, 2, 1024, 64, 17, skip_rate=0.5, block=128)
    plain = wl.layer_inputs(2, 2, 1024, 64, 17)
    assert x.skip_tier.shape == (2, 8) and not x.skip_tier[:, 0].any()
    assert 0 < int(x.skip_tier.sum()) < 16
    for kh in range(2):
        for j in range(8):
            blk, ref = x.k[kh, j * 128:(j + 1) * 128].float(), plain.k[kh, j * 128:(j + 1) * 128].float()
            r = float(blk.norm() / ref.norm())
            assert abs(r - (0.01 if x.skip_tier[kh, j] else 1.0)) < 0.01 * (0.01 if x.skip_tier[kh, j] else 1.0) + 1e-3


def test_workload_shapes_and_visible_tiles():
    """The five benchmark workloads keep their stated shapes, and their
    visible-tile counts (counted block by block with the oracle's geometry)
    equal the closed form Hq * sum_b n_b (n_b + 1) / 2: 272 for the tiny case,
    1,052,672 at 32K, 16,793,600 at 128K, 4,202,496 at 64K and 8,710,144 per
    layer for the 8-sequence batch."""
    from oracle import bsfa_oracle as orc
    W = wl.WORKLOADS
    assert (W["tiny-h2-d64-L1024"]["Hq"], W["tiny-h2-d64-L1024"]["d"],
            W["tiny-h2-d64-L1024"]["L"], W["tiny-h2-d64-L1024"]["Bq"]) == (2, 64, 1024, 64)
    for name in ("llama8b-L32768", "llama8b-L131072", "lambda-sweep-L65536",
                 "varlen-8seq-32layer"):
        c = W[name]
        assert (c["Hq"], c["Hkv"], c["d"], c["Bq"], c["Bk"]) == (32, 8, 128, 128, 128), name
    assert W["llama8b-L131072"]["ks"] == [32, 128, 512]
    assert W["llama8b-L131072"]["cal_L"] == 65536
    assert W["varlen-8seq-32layer"]["lens"] == [n * 1024 for n in (4, 8, 12, 16, 24, 32, 48, 64)]
    stated = {"tiny-h2-d64-L1024": 272, "llama8b-L32768": 1_052_672,
              "llama8b-L131072": 16_793_600, "lambda-sweep-L65536": 4_202_496,
              "varlen-8seq-32layer": 8_710_144}
    for name, want in stated.items():
        c = W[name]
        lens = c.get("lens", [c.get("L")])
        per_head = 0
        for Ln in lens:
            n = orc.num_blocks(Ln, c["Bq"])
            per_head += sum(1 for i in range(n) for j in range(orc.num_blocks(Ln, c["Bk"]))
                            if orc.block_class(i, j, c["Bq"], c["Bk"], Ln) is not None)
        assert c["Hq"] * per_head == want, name
        assert want == c["Hq"] * sum(orc.num_blocks(Ln, c["Bq"]) * (orc.num_blocks(Ln, c["Bq"]) + 1)
                                     // 2 for Ln in lens)
