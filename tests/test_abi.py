"""The C ABI library builds, loads without a GPU, and exports every entry
point ``include/pa.h`` and ``include/pa_testing.h`` declare; the Python binding declares each with the
header's argument count.  The native block manager matches the oracle's
model op for op (statuses, ids, slots, copy requests, refcounts)."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in ("pa.h", "pa_testing.h")]


@pytest.fixture(scope="session")
def palib():
    from paged_kv_cache_228_gb300 import build, pa
    build.build()
    return pa


def _declared():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for m in re.finditer(r"\b(pa_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        name, args = m.group(1), m.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        decls[name] = n
    return decls


def test_header_declares_the_boundary():
    d = _declared()
    for name in ("pa_cache_write", "pa_decode", "pa_copy_blocks", "pa_quantize_fp8",
                 "pa_decode_workspace_size", "pa_block_alloc", "pa_block_free",
                 "pa_block_fork", "pa_seq_append_slots", "pa_get_device_error"):
        assert name in d, name


def test_library_exports_every_declared_symbol(palib):
    L = palib.lib()
    for name in _declared():
        assert hasattr(L, name), f"libpa.so does not export {name}"


def test_binding_signatures_match_header(palib):
    d = _declared()
    assert set(d) == set(palib.SIGNATURES), set(d) ^ set(palib.SIGNATURES)
    for name, n in d.items():
        assert len(palib.SIGNATURES[name][1]) == n, name


def test_status_strings(palib):
    assert palib.status_string(0) == "PA_OK"
    assert palib.status_string(6) == "PA_ERR_WORKSPACE"
    assert palib.pa_abi_version() == 1


def test_host_validation_without_gpu(palib):
    # Invalid arguments are rejected on the host before any CUDA call.
    L = palib.lib()
    assert L.pa_decode(None, None, None, None, None, 0, None, 1, None, 1, 4, 3, 64, 16,
                       8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_decode(None, None, None, None, None, 0, None, 1, None, 1, 32, 2, 64, 16,
                       8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_cache_write(None, None, None, 1, None, None, 1, 1, 16, 64,
                            palib.PA_KV_FP8_E4M3, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_cache_write(None, None, None, 0, None, None, 1, 1, 16, 64,
                            palib.PA_KV_BF16, None) == palib.PA_OK
    # fused append: missing new-token buffers, unsupported shapes
    assert L.pa_decode_append(None, None, None, None, None, None, None, 1, None, 1, 4, 2, 64,
                              16, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_decode_append(None, None, None, None, None, None, None, 1, None, 1, 4, 2, 96,
                              16, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_decode_append(None, None, None, None, None, None, None, 1, None, 0, 4, 2, 64,
                              16, 8, 1.0, None, None, 0, 0, None) == palib.PA_OK
    # swap: missing buffers are rejected before any CUDA call
    assert L.pa_swap_out(None, None, None, None, None, 3, None, None, None, None, 8, 2, 16, 64,
                         palib.PA_KV_BF16, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_swap_in(None, None, None, None, None, 0, None, None, None, None, 8, 2, 16, 64,
                        palib.PA_KV_BF16, None) == palib.PA_OK
    # cascade: the prefix must be a multiple of 16 and of the block size
    assert L.pa_decode_cascade(None, None, None, None, 8, None, 1, 4, 2, 64, 16, 8, 24, 1.0,
                               None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_decode_cascade(None, None, None, None, 8, None, 1, 4, 2, 64, 32, 8, 16, 1.0,
                               None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    # NVFP4: tensor scales must be positive and finite; block_size >= 16
    nan, inf = float("nan"), float("inf")
    for gs in (0.0, -1.0, nan, inf):
        assert L.pa_cache_write_nvfp4(None, None, None, 1, None, None, None, None, gs, 1.0, 8,
                                      2, 16, 64, None) == palib.PA_ERR_INVALID_ARG
        assert L.pa_decode_nvfp4(None, None, None, None, None, 1.0, gs, None, 1, None, 1, 4, 2,
                                 64, 16, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_cache_write_nvfp4(None, None, None, 1, None, None, None, None, 1.0, 1.0, 8, 2,
                                  8, 64, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_cache_write_nvfp4(None, None, None, 1, None, None, None, None, 1.0, 1.0, 8, 2,
                                  16, 96, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_cache_write_nvfp4(None, None, None, 0, None, None, None, None, 1.0, 1.0, 8, 2,
                                  16, 64, None) == palib.PA_OK
    assert L.pa_cache_write_nvfp4(None, None, None, 3, None, None, None, None, 1.0, 1.0, 8, 2,
                                  16, 64, None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_decode_nvfp4(None, None, None, None, None, 1.0, 1.0, None, 1, None, 1, 32, 2,
                             64, 16, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_decode_nvfp4(None, None, None, None, None, 1.0, 1.0, None, 1, None, 1, 4, 2,
                             64, 8, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_UNSUPPORTED
    assert L.pa_decode_nvfp4(None, None, None, None, None, 1.0, 1.0, None, 1, None, 0, 4, 2,
                             64, 16, 8, 1.0, None, None, 0, 0, None) == palib.PA_OK
    assert L.pa_decode_nvfp4(None, None, None, None, None, 1.0, 1.0, None, 1, None, 1, 4, 2,
                             64, 16, 8, 1.0, None, None, 0, 0, None) == palib.PA_ERR_INVALID_ARG
    # fused NVFP4 append: the new-token buffers are required
    assert L.pa_decode_append_nvfp4(None, None, None, None, None, None, None, None, 1.0, 1.0,
                                    None, 1, None, 1, 4, 2, 64, 16, 8, 1.0, None, None, 0, 0,
                                    None) == palib.PA_ERR_INVALID_ARG
    assert L.pa_decode_append_nvfp4(None, None, None, None, None, None, None, None, 1.0, 1.0,
                                    None, 1, None, 0, 4, 2, 64, 16, 8, 1.0, None, None, 0, 0,
                                    None) == palib.PA_OK


def _compare_models(pa, seed, steps=2000, N=48, bs=4):
    from oracle import block_manager as BM
    rng = np.random.default_rng(seed)
    m = BM.BlockManagerModel(N)
    a = pa.Allocator(N)
    seqs_m, seqs_a = {}, {}
    for step in range(steps):
        op = int(rng.integers(0, 5))
        if op <= 1 or not seqs_m:
            sid = int(rng.integers(0, 10))
            tm, nm = seqs_m.get(sid, ([], 0))
            ta, na = seqs_a.get(sid, ([], 0))
            k = int(rng.integers(0, 7))
            st1, s1, p1 = m.append_slots(tm, nm, k, bs, 24)
            st2, s2, p2 = a.append_slots(ta, na, k, bs, 24)
            assert st1 == st2 and s1 == s2 and p1 == p2, (step, st1, st2)
            if st1 == BM.OK:
                seqs_m[sid], seqs_a[sid] = (tm, nm + k), (ta, na + k)
                assert tm == ta
        elif op == 2:
            sid = list(seqs_m)[int(rng.integers(0, len(seqs_m)))]
            new = 1000 + step
            st1, st2 = m.fork(seqs_m[sid][0]), a.fork(seqs_a[sid][0])
            assert st1 == st2
            if st1 == BM.OK:
                seqs_m[new] = (list(seqs_m[sid][0]), seqs_m[sid][1])
                seqs_a[new] = (list(seqs_a[sid][0]), seqs_a[sid][1])
        elif op == 3:
            sid = list(seqs_m)[int(rng.integers(0, len(seqs_m)))]
            t, _ = seqs_m.pop(sid)
            seqs_a.pop(sid)
            assert m.free(t) == a.free(t) == BM.OK
        else:
            # error paths: ids outside the pool, freeing / forking a free
            # block, oversize alloc; none may change either state
            bad = [int(rng.choice([-3, -1, N, N + 2]))]
            if m.num_free():
                bad.append(m.free_stack[-1])
            for x in bad:
                assert m.free([x]) == a.free([x]) == BM.BAD_BLOCK_ID
                assert m.fork([x]) == a.fork([x]) == BM.BAD_BLOCK_ID
            n = int(rng.integers(0, N + 2))
            st1, ids1 = m.alloc(n)
            st2, ids2 = a.alloc(n)
            assert st1 == st2 and ids1 == ids2
            if st1 == BM.OK:
                assert m.free(ids1) == a.free(ids2) == BM.OK
        assert m.num_free() == a.num_free()
    for bid in range(N):
        assert (BM.OK, m.refcount[bid]) == a.refcount(bid)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_native_block_manager_matches_model(palib, seed):
    _compare_models(palib, seed)


def test_native_replay_matches_model_on_workloads(palib):
    from oracle import block_manager as BM
    from paged_kv_cache_228_gb300 import workloads as W
    for name in ("tiny", "llama3.2-1b", "llama3.1-8b", "shared_prefix_bs16"):
        w = W.WORKLOADS[name]()
        ops = W.build_script(w)
        _, t1, l1 = BM.replay_script(ops, w.num_seqs, w.block_size, w.max_blocks_per_seq,
                                     w.pool_blocks)
        a, t2, l2 = palib.replay_script(ops, w.num_seqs, w.block_size, w.max_blocks_per_seq,
                                        w.pool_blocks)
        assert t1 == t2 and l1 == l2, name


def test_batch_append_matches_model(palib):
    # One native call per step against the oracle's model appending the
    # same batch sequence by sequence; a step that runs out of blocks stops
    # at the failing sequence and leaves it and later ones untouched.
    from oracle import block_manager as BM
    pa = palib
    rng = np.random.default_rng(11)
    N, bs, maxb, B = 40, 4, 16, 9
    m = BM.BlockManagerModel(N)
    a = pa.Allocator(N)
    tm = [[] for _ in range(B)]
    ba = pa.BatchAppender(a, tm, maxb)
    lens = np.zeros(B, dtype=np.int32)
    saw_stop = False
    for step in range(60):
        n_new = rng.integers(0, 4, size=B).astype(np.int32)
        if step % 7 == 3:           # fork a sequence into another slot's place
            src, dst = rng.integers(0, B, size=2)
            if src != dst and lens[src] > 0:
                m.free(tm[dst]); assert a.free(list(ba.tables[dst][ba.tables[dst] >= 0])) == 0
                tm[dst] = list(tm[src]); ba.tables[dst] = ba.tables[src]
                assert m.fork(tm[dst]) == 0 and a.fork(tm[dst]) == 0
                lens[dst] = lens[src]
        st, slots, pairs, done = ba.append(lens, n_new, bs)
        ms, mp, mdone, mst = [], [], 0, BM.OK
        for i in range(B):
            st_i, s_i, p_i = m.append_slots(tm[i], int(lens[i]), int(n_new[i]), bs, maxb)
            if st_i != BM.OK:
                mst = st_i
                break
            ms += s_i; mp += p_i; mdone = i + 1
        assert (st, done) == (mst, mdone), step
        assert list(slots) == ms and pairs == mp, step
        for i in range(B):
            assert list(ba.tables[i][:len(tm[i])]) == tm[i] and \
                (ba.tables[i][len(tm[i]):] == -1).all(), (step, i)
        lens[:done] += n_new[:done]
        if st != 0:
            saw_stop = True
            # finish some sequences to make room again
            for i in range(0, B, 2):
                assert m.free(tm[i]) == 0
                assert a.free(list(ba.tables[i][ba.tables[i] >= 0])) == 0
                tm[i] = []; ba.tables[i] = -1; lens[i] = 0
    assert saw_stop


@pytest.mark.parametrize("name", ["tiny", "llama3.1-8b", "shared_prefix_bs8"])
def test_allocator_usage_matches_model(palib, name):
    # the fragmentation report of a workload's pre-step state, native vs model
    from oracle import block_manager as BM
    from paged_kv_cache_228_gb300 import workloads as W
    w = W.WORKLOADS[name]()
    ops = W.build_script(w)
    maxb = w.max_blocks_per_seq
    m, tm, lm = BM.replay_script(ops, w.num_seqs, w.block_size, maxb, w.pool_blocks)
    a, ta, la = palib.replay_script(ops, w.num_seqs, w.block_size, maxb, w.pool_blocks)
    assert palib.allocator_usage(a, ta, la, w.block_size) == BM.usage(m, tm, lm, w.block_size)


def test_wait_limit_hook_validates_on_the_host(palib):
    # The bounded-wait test hook (include/pa_testing.h): host-side settings
    # only, no CUDA call; 0 polls restores the default.
    L = palib.lib()
    assert L.pa_testing_set_wait_limit(100, 2) == palib.PA_ERR_INVALID_ARG
    assert L.pa_testing_set_wait_limit(100, 1) == palib.PA_OK
    assert L.pa_testing_set_wait_limit(0, 1) == palib.PA_OK
