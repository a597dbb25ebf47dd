"""Host-side byte accounting, pinned by the worked example the pages print."""
import json
import os

import numpy as np

from paged_kv_cache_265_gb300 import workload as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kv_bytes_worked_examples.json")))


def test_opt13b_worked_example():
    g = GOLD["opt13b"]
    # OPT-13B: 40 heads x 128 = 5120 hidden, 40 layers, fp16
    per_tok = W.kv_bytes_per_token(g["num_layers"], 40, 128, g["elem_bytes"])
    assert 40 * 128 == g["hidden"]
    assert per_tok == g["kv_bytes_per_token"]
    assert per_tok // 1024 == g["kv_bytes_per_token_kib"]
    assert round(per_tok * g["max_tokens"] / 2 ** 30, 1) == g["request_gb_rounded"]


def test_block_bytes_is_block_size_tokens_of_one_layer():
    assert W.BLOCK_SIZE == GOLD["default_block_size"]
    for hkv, d in [(8, 128), (40, 128), (4, 64)]:
        assert W.block_bytes(16, hkv, d, 2) == 16 * W.kv_bytes_per_token(1, hkv, d, 2)


def test_attention_bytes_counts_every_position_once():
    w = W.make_workload("b", [2, 17, 100], num_heads=8, num_kv_heads=2, head_dim=64, q_len=2,
                        num_blocks=16, seed=1)
    kv = (2 + 17 + 100) * 2 * 2 * 64 * 2
    qo = 2 * 3 * 2 * 8 * 64 * 2
    assert W.attention_bytes(w) == kv + qo
    assert W.append_bytes(w) == 2 * (3 * 2) * 2 * 2 * 64 * 2


def test_workloads_are_seeded_and_shaped():
    a = W.tiny_mha(keep_logical=True)
    b = W.tiny_mha(keep_logical=True)
    assert np.array_equal(a.key_cache, b.key_cache) and np.array_equal(a.query, b.query)
    assert list(a.context_lens) == [1, 17, 33, 100]
    assert a.slot_mapping.shape == (4,) and a.new_key.shape == (4, 4, 64)
    # every used block id is distinct and inside the 64-block pool
    used = a.block_tables[a.block_tables >= 0]
    assert len(set(used.tolist())) == used.size and used.max() < 64
    # unused slots hold the NaN sentinel
    assert a.key_cache[a.block_tables[0, 0], 1, 0, 0] == W.NAN_BITS["bf16"]


def test_unique_bytes_count_shared_blocks_once():
    """Shared prefix: the 64 common blocks count once in the unique bytes; without sharing the
    unique and logical bytes agree."""
    w = W.shared_prefix_verify()
    logical, unique = W.attention_bytes(w), W.unique_attention_bytes(w)
    per_token = W.kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, 2)
    shared_rows = w.shared_prefix_blocks * w.block_size
    assert logical - unique == (w.num_seqs - 1) * shared_rows * per_token
    t = W.tiny_mha()
    assert W.unique_attention_bytes(t) == W.attention_bytes(t)
