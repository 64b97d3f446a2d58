"""Model of the host-side block manager (oracle; test infrastructure only).

The page "Paged Attention and KV Cache Fragmentation", section "How
PagedAttention maps an OS concept onto GPU memory", fixes the behaviour:

* the pool is cut into fixed-size blocks; any freed block fits any request;
* a sequence gets a new block only when it actually grows past its last one;
* a finished request's blocks are freed at once;
* sequences with a shared prefix (system prompt, beam branches, tool-use
  forks; also the "KV cache fragmentation" field guide, section "Why it
  matters") point at the same physical blocks and diverge only where their
  content differs.

The pages leave the free-list order, error handling and the copy-on-write
mechanics open.  Readings taken here (and implemented identically by the
native manager, which the tests check op for op):

* the free list is a LIFO stack that initially pops 0, 1, 2, ...;
* every call is all-or-nothing: on any error nothing changes;
* ``free`` decrements a refcount and returns the block at zero; freeing a
  block more times than it is referenced is an error;
* ``fork`` increments refcounts of live blocks (the child shares them);
* ``append_slots`` first copies a shared, partially filled tail block into a
  fresh block (copy-on-write: one (src, dst, valid_slots) copy request), then
  allocates blocks for every block boundary the new tokens cross, and returns
  each new token's flat slot ``block * block_size + offset``.
"""
from __future__ import annotations

OK, INVALID_ARG, OUT_OF_BLOCKS, BAD_BLOCK_ID = 0, 1, 2, 3


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


class BlockManagerModel:
    def __init__(self, num_blocks: int):
        if num_blocks < 0:
            raise ValueError("num_blocks < 0")
        self.num_blocks = num_blocks
        self.refcount = [0] * num_blocks
        self.free_stack = list(range(num_blocks - 1, -1, -1))  # pop() -> 0, 1, ...

    # -------------------------------------------------------------- queries
    def num_free(self) -> int:
        return len(self.free_stack)

    def get_refcount(self, bid: int):
        if not (0 <= bid < self.num_blocks):
            return BAD_BLOCK_ID, None
        return OK, self.refcount[bid]

    # ----------------------------------------------------------- mutations
    def alloc(self, n: int):
        if n < 0:
            return INVALID_ARG, None
        if n > len(self.free_stack):
            return OUT_OF_BLOCKS, None
        ids = [self.free_stack.pop() for _ in range(n)]
        for i in ids:
            self.refcount[i] = 1
        return OK, ids

    def free(self, ids):
        need = {}
        for i in ids:
            if not (0 <= i < self.num_blocks):
                return BAD_BLOCK_ID
            need[i] = need.get(i, 0) + 1
        for i, c in need.items():
            if self.refcount[i] < c:
                return BAD_BLOCK_ID
        for i in ids:
            self.refcount[i] -= 1
            if self.refcount[i] == 0:
                self.free_stack.append(i)
        return OK

    def fork(self, ids):
        for i in ids:
            if not (0 <= i < self.num_blocks) or self.refcount[i] <= 0:
                return BAD_BLOCK_ID
        for i in ids:
            self.refcount[i] += 1
        return OK

    def append_slots(self, table, length: int, n: int, block_size: int,
                     max_blocks: int):
        """Grow one sequence from ``length`` to ``length + n`` tokens.

        ``table`` is a list of physical block ids (modified in place on
        success).  Returns (status, slots, cow_pairs).
        """
        if length < 0 or n < 0 or block_size <= 0:
            return INVALID_ARG, None, None
        held = _cdiv(length, block_size)
        want = _cdiv(length + n, block_size)
        if want > max_blocks or held > len(table):
            return INVALID_ARG, None, None
        for j in range(held):
            b = table[j]
            if not (0 <= b < self.num_blocks) or self.refcount[b] <= 0:
                return BAD_BLOCK_ID, None, None
        cow = (n > 0 and length % block_size != 0
               and self.refcount[table[held - 1]] > 1)
        if (want - held) + (1 if cow else 0) > len(self.free_stack):
            return OUT_OF_BLOCKS, None, None
        while len(table) < want:
            table.append(-1)
        pairs = []
        if cow:
            old = table[held - 1]
            new = self.free_stack.pop()
            self.refcount[new] = 1
            self.refcount[old] -= 1
            table[held - 1] = new
            pairs.append((old, new, length % block_size))
        for j in range(held, want):
            b = self.free_stack.pop()
            self.refcount[b] = 1
            table[j] = b
        slots = [table[p // block_size] * block_size + p % block_size
                 for p in range(length, length + n)]
        return OK, slots, pairs


def replay_script(ops, num_seqs: int, block_size: int, max_blocks: int,
                  num_blocks: int):
    """Apply a workload op script (see the workloads module) to a fresh model.

    Returns (model, tables, lens): per-sequence block-id lists and token
    counts after the script.  Raises on any non-OK status.
    """
    m = BlockManagerModel(num_blocks)
    tables = [[] for _ in range(num_seqs)]
    lens = [0] * num_seqs
    for op in ops:
        kind = op[0]
        if kind == "alloc":
            st, ids = m.alloc(op[1])
            assert st == OK, ("alloc", st)
        elif kind == "free_list":
            st = m.free(op[1])
            assert st == OK, ("free", st)
        elif kind == "append":
            _, b, n = op
            st, _, _ = m.append_slots(tables[b], lens[b], n, block_size,
                                      max_blocks)
            assert st == OK, ("append", b, st)
            lens[b] += n
        elif kind == "fork":
            _, child, parent, ntok = op
            ids = tables[parent][:_cdiv(ntok, block_size)]
            st = m.fork(ids)
            assert st == OK, ("fork", st)
            tables[child] = list(ids)
            lens[child] = ntok
        else:
            raise ValueError(kind)
    return m, tables, lens


# ------------------------------------------------------- usage report ---
# The pages' fragmentation argument ("KV cache fragmentation" field guide,
# section "Why it matters"; "Paged Attention and KV Cache Fragmentation",
# section "How PagedAttention maps an OS concept onto GPU memory"): a paged
# cache wastes at most the unfilled tail of each sequence's last block,
# where a contiguous cache reserves each request's maximum length up front.
# The report counts, for a set of sequences (tables + lengths):
#   live_blocks     blocks with a nonzero refcount
#   slots_reserved  live_blocks * block_size
#   tokens_stored   distinct (block, offset) slots holding a token of some
#                   sequence (a shared block counted once)
#   tokens_logical  sum of the sequence lengths


def usage(model: BlockManagerModel, tables, lens, block_size: int) -> dict:
    live = sum(1 for r in model.refcount if r > 0)
    held = set()
    for t, n in zip(tables, lens):
        for p in range(int(n)):
            held.add((t[p // block_size], p % block_size))
    return {"live_blocks": live, "slots_reserved": live * block_size,
            "tokens_stored": len(held), "tokens_logical": int(sum(int(n) for n in lens))}
