"""Pins for the oracle's block-manager model.

* LIFO order and all-or-nothing allocation, written out by hand;
* conservation: free + distinct live blocks == pool size, and every live
  block's refcount equals the number of tables holding it, under random
  seeded op sequences;
* errors (double free, bad ids, out of blocks) leave the state unchanged;
* copy-on-write fires exactly when a shared block is partially filled;
* the footprint formula reproduces the page's 70B / 128K numbers.
"""
import copy
import os

import numpy as np

from oracle import block_manager as BM
from oracle import footprint

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_footprint_70b_128k.txt")


def test_lifo_order_by_hand():
    m = BM.BlockManagerModel(5)
    assert m.alloc(3) == (BM.OK, [0, 1, 2])
    assert m.free([1]) == BM.OK
    assert m.alloc(1) == (BM.OK, [1])
    assert m.free([2, 0]) == BM.OK
    assert m.alloc(3) == (BM.OK, [0, 2, 3])
    assert m.num_free() == 1


def test_all_or_nothing_and_errors():
    m = BM.BlockManagerModel(4)
    st, ids = m.alloc(3)
    snap = copy.deepcopy(m.__dict__)
    assert m.alloc(2) == (BM.OUT_OF_BLOCKS, None)
    assert m.free([0, 0]) == BM.BAD_BLOCK_ID          # more frees than refs
    assert m.free([7]) == BM.BAD_BLOCK_ID
    assert m.fork([3]) == BM.BAD_BLOCK_ID             # 3 is free
    assert m.alloc(-1) == (BM.INVALID_ARG, None)
    assert m.__dict__ == snap
    assert m.fork([0]) == BM.OK and m.free([0, 0]) == BM.OK
    assert m.free([0]) == BM.BAD_BLOCK_ID


def test_append_allocates_only_on_block_boundaries():
    m = BM.BlockManagerModel(10)
    table = []
    st, slots, pairs = m.append_slots(table, 0, 5, 4, 8)
    assert st == BM.OK and table == [0, 1] and slots == [0, 1, 2, 3, 4]
    st, slots, pairs = m.append_slots(table, 5, 3, 4, 8)
    assert table == [0, 1] and slots == [5, 6, 7] and pairs == []
    st, slots, pairs = m.append_slots(table, 8, 1, 4, 8)
    assert table == [0, 1, 2] and slots == [8]
    assert m.append_slots(table, 9, 40, 4, 8)[0] == BM.INVALID_ARG


def test_copy_on_write_of_shared_partial_tail():
    m = BM.BlockManagerModel(8)
    parent = []
    m.append_slots(parent, 0, 6, 4, 4)                  # blocks [0, 1], 6 tokens
    child = list(parent)
    assert m.fork(child) == BM.OK
    st, slots, pairs = m.append_slots(child, 6, 1, 4, 4)
    assert st == BM.OK and pairs == [(1, 2, 2)]
    assert child == [0, 2] and parent == [0, 1] and slots == [2 * 4 + 2]
    assert m.get_refcount(1) == (BM.OK, 1) and m.get_refcount(0) == (BM.OK, 2)
    # the last holder appends in place: no copy
    st, slots, pairs = m.append_slots(parent, 6, 1, 4, 4)
    assert pairs == [] and slots == [1 * 4 + 2]
    # a full shared block needs no copy: the next token opens a new block
    p2 = []
    m.append_slots(p2, 0, 4, 4, 4)
    m.fork(p2)
    st, slots, pairs = m.append_slots(list(p2), 4, 1, 4, 4)
    assert pairs == []


def test_out_of_blocks_append_changes_nothing():
    m = BM.BlockManagerModel(3)
    t = []
    m.append_slots(t, 0, 8, 4, 4)
    m.fork(t)
    snap = copy.deepcopy(m.__dict__)
    t2 = list(t)
    assert m.append_slots(t2, 8, 5, 4, 4)[0] == BM.OUT_OF_BLOCKS
    assert m.__dict__ == snap and t2 == t


def test_conservation_under_random_ops():
    rng = np.random.default_rng(0)
    N, bs = 64, 4
    m = BM.BlockManagerModel(N)
    seqs = {}
    for step in range(3000):
        op = rng.integers(0, 4)
        if op == 0 or not seqs:                      # new or grow
            sid = int(rng.integers(0, 12))
            t, n = seqs.get(sid, ([], 0))
            k = int(rng.integers(1, 9))
            st, _, _ = m.append_slots(t, n, k, bs, 32)
            if st == BM.OK:
                seqs[sid] = (t, n + k)
        elif op == 1:                                # fork
            sid = list(seqs)[int(rng.integers(0, len(seqs)))]
            t, n = seqs[sid]
            new = 100 + step
            if m.fork(t) == BM.OK:
                seqs[new] = (list(t), n)
        else:                                        # finish
            sid = list(seqs)[int(rng.integers(0, len(seqs)))]
            t, n = seqs.pop(sid)
            assert m.free(t) == BM.OK
        holders = {}
        for t, _ in seqs.values():
            for b in t:
                holders[b] = holders.get(b, 0) + 1
        assert m.num_free() + len(holders) == N
        for b in range(N):
            assert m.refcount[b] == holders.get(b, 0)


def test_footprint_matches_page_numbers():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        L, H, d, T, s2, gb = line.split()
        b = int(T) * footprint.kv_bytes_per_token(int(L), int(H), int(d), 1) * int(s2) // 2
        assert round(b / 1e9, 1) == float(gb)
    # one layer of the 70B / 128K request, bf16: exactly 2 * 8 * 128 * 131072 * 2
    assert footprint.decode_step_kv_bytes([131072], 8, 128, 2) == 536870912


def test_usage_closed_forms():
    # B private sequences of length n: ceil(n / bs) blocks each, n tokens each
    bs, B, n = 16, 5, 37
    m = BM.BlockManagerModel(64)
    tables = []
    for _ in range(B):
        t = []
        assert m.append_slots(t, 0, n, bs, 8)[0] == BM.OK
        tables.append(t)
    u = BM.usage(m, tables, [n] * B, bs)
    assert u == {"live_blocks": B * 3, "slots_reserved": B * 48, "tokens_stored": B * n,
                 "tokens_logical": B * n}
    # a shared 32-token prefix (2 full blocks) forked into 4 children that
    # each add r tokens: stored = 32 + sum(r), logical = 4 * 32 + sum(r)
    m = BM.BlockManagerModel(64)
    parent = []
    m.append_slots(parent, 0, 32, bs, 8)
    kids, lens = [], []
    for r in (1, 16, 17, 5):
        t = list(parent)
        m.fork(t)
        assert m.append_slots(t, 32, r, bs, 8)[0] == BM.OK
        kids.append(t)
        lens.append(32 + r)
    m.free(parent)
    u = BM.usage(m, kids, lens, bs)
    assert u["tokens_stored"] == 32 + 1 + 16 + 17 + 5
    assert u["tokens_logical"] == 4 * 32 + 39
    assert u["live_blocks"] == 2 + (1 + 1 + 2 + 1)
    assert u["slots_reserved"] == u["live_blocks"] * bs


def test_footprint_fp8_scale_bytes_closed_forms():
    # The FP8 branch: codes at one byte per value plus two fp32 scales (K, V)
    # per (block, KV head) a sequence touches.  70B layer at 128K, 8
    # sequences: 2^31 code bytes and 2 * 8192 blocks * 8 heads * 4 B * 8.
    n = [131072] * 8
    assert footprint.decode_step_kv_bytes(n, 8, 128, 1, 16, 4) == 2 ** 31 + 2 * 8 * 8192 * 8 * 4
    assert footprint.decode_step_kv_bytes(n, 8, 128, 1, 16, 4) == 2151677952
    # worked by hand: 17 tokens in 16-token blocks touch 2 blocks; 2 heads,
    # d = 64: 17 * 2 * 2 * 64 = 4352 code bytes + 2 * 2 * 2 * 4 = 32 scale bytes
    assert footprint.decode_step_kv_bytes([17], 2, 64, 1, 16, 4) == 4384
    # an exact block multiple adds no partial block; length 0 touches none
    assert footprint.decode_step_kv_bytes([32, 0], 2, 64, 1, 16, 4) == 32 * 256 + 2 * 2 * 2 * 4
    # without scales the branch is the plain footprint
    assert footprint.decode_step_kv_bytes([17], 2, 64, 1, 16, 0) == 4352


def test_bench_byte_counts_equal_the_oracle_footprint():
    # bench.py restates the algorithmic byte counts (the product must not
    # import the oracle); they must equal the pinned oracle functions on
    # every workload and format.
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from paged_kv_cache_228_gb300 import workloads as W
    for name, make in W.WORKLOADS.items():
        w = make()
        H, d, bs = w.num_kv_heads, w.head_dim, w.block_size
        assert bench.kv_bytes(w) == footprint.decode_step_kv_bytes(w.seq_lens, H, d, 2), name
        assert bench.kv_bytes(w, 1, 4) == footprint.decode_step_kv_bytes(
            w.seq_lens, H, d, 1, bs, 4), name
        assert bench.kv_bytes_nvfp4(w) == sum(w.seq_lens) * footprint.nvfp4_bytes_per_token(
            1, H, d), name
    assert bench.kv_bytes(W.llama31_70b_128k(), 1, 4) == 2151677952
