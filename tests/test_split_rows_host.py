"""Host logic of split-QKV (Megatron-LM issue #6720: NS per Q, K, V block):
the row-block views a fused QKV projection is split into."""

import torch

import workloads


def test_blocks_tile_each_parent_exactly():
    for w in (workloads.gpt_24l_d2048(), workloads.llama8b_32l()):
        shapes = w.shapes[:5]
        blocks, parents = workloads.split_rows(shapes)
        rows = {}
        for b, (i, r0) in zip(blocks, parents):
            assert tuple(b[1:]) == tuple(shapes[i][1:])
            assert r0 == rows.get(i, 0)          # blocks follow each other, no gap or overlap
            rows[i] = r0 + b[0]
        assert all(rows[i] == shapes[i][0] for i in range(len(shapes)))


def test_llama_gqa_blocks_and_untouched_shapes():
    blocks, parents = workloads.split_rows([(6144, 4096), (4096, 4096)])
    assert blocks == [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096)]
    assert parents == [(0, 0), (0, 4096), (0, 5120), (1, 0)]


def test_block_views_reassemble_the_tensor():
    t = torch.arange(6 * 3).reshape(6, 3)
    blocks, parents = workloads.split_rows([(6, 3)], {(6, 3): (2, 1, 3)})
    views = [t[r0:r0 + b[0]] for b, (_, r0) in zip(blocks, parents)]
    assert torch.equal(torch.cat(views), t)
