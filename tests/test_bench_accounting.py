"""The bench's byte accounting (the numerator of every roofline fraction),
checked on hand-sized cases on the CPU.

Algorithmic bytes of one decode step: each cluster's mean key and value sum
(index bytes per element) with its size, once; the steady zone's K and V rows;
the retrieved clusters' K and V rows, once per (sequence, KV head, cluster)
whichever query heads of the group picked them."""

from types import SimpleNamespace

import torch

import bench

ROW = 128 * 2 * 2  # one token's K and V rows, bf16, d = 128


def test_retrieved_rows_counted_once_per_group():
    # B = 1, Hq = 4, G = 2 (two KV groups), r = 3, -1 padding
    size = torch.tensor([[[5, 7, 0, 2], [1, 1, 4, 9]]], dtype=torch.int32)
    topk = torch.tensor([[[0, 1, -1],    # group 0, head 0
                          [1, 3, -1],    # group 0, head 1: cluster 1 again
                          [2, 3, -1],    # group 1, head 0
                          [2, -1, -1]]], dtype=torch.int32)
    # group 0 reads clusters {0, 1, 3}: 5 + 7 + 2 tokens; group 1 {2, 3}: 4 + 9
    assert bench.retrieved_unique_bytes(topk, size, 2) == (14 + 13) * ROW
    # G = 1: every head is its own group (Hkv = 4) and reads its own KV
    # head's sizes: {0, 1} -> 5 + 7, {1, 3} -> 1 + 9, {2, 3} -> 3 + 3, {2} -> 0
    size4 = torch.tensor([[[5, 7, 0, 2], [1, 1, 4, 9], [3, 3, 3, 3], [8, 0, 0, 0]]],
                         dtype=torch.int32)
    assert bench.retrieved_unique_bytes(topk, size4, 1) == (12 + 10 + 6 + 0) * ROW


def test_step_bytes_hand_count():
    w = SimpleNamespace(n_clusters=3, B=2, Hq=4, Hkv=2, d=128, sink=4, window=12)
    ix = SimpleNamespace(size=torch.tensor([[[2, 0, 5], [1, 1, 1]], [[0, 0, 9], [4, 4, 0]]],
                                           dtype=torch.int32))
    topk = torch.tensor([[[2, -1], [0, 2], [0, 1], [2, -1]],
                         [[2, -1], [-1, -1], [1, -1], [0, 1]]], dtype=torch.int32)
    by = bench.decode_bytes(w, ix, topk, 2)
    # 2 sequences x 2 KV heads x 3 clusters, 128 f32 and one i32 size each
    assert by["centroid_keys"] == 12 * (512 + 4)
    assert by["value_sums_sizes"] == 12 * (512 + 4)
    # 16 steady tokens per (sequence, KV head)
    assert by["steady_kv"] == 4 * 16 * ROW
    # (b0, g0): {0, 2} -> 2 + 5; (b0, g1): {0, 1, 2} -> 3; (b1, g0): {2} -> 9;
    # (b1, g1): {0, 1} -> 8
    assert by["retrieved_kv_unique"] == (7 + 3 + 9 + 8) * ROW
    # bf16 index: half the index elements' bytes, sizes unchanged
    by16 = bench.decode_bytes(w, ix, topk, 2, index_bytes=2)
    assert by16["centroid_keys"] == 12 * (256 + 4)
    # no budget: nothing retrieved
    assert bench.decode_bytes(w, ix, topk, 0)["retrieved_kv_unique"] == 0
