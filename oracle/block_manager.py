"""KV cache manager: block allocator, reference counts, fork / append / free and the
copy-on-write decision, in plain Python.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only ``tests/`` and the
CPU-baseline leg of ``bench.py`` may use it; the library never imports it.

What it follows (sources are the web pages on the subject):

* vLLM post (devpress), "1. overall architecture", KV cache manager and block
  engine: the pool is cut into equal physical blocks; a request is a list of
  logical blocks filled left to right; the block table maps each logical block to a
  physical block and keeps the number of filled slots of the last one; a new
  physical block is taken only when the last logical block is full (worked example:
  a 7-token prompt with block size 4 in physical blocks 7 and 1, #filled 3 -> 4 at
  the first decode step, a new physical block 3 at the second); a finished request's
  blocks are freed.
* Same post, "2.1 parallel sampling": samples of one prompt share its physical
  blocks, each of which carries a reference count; a sample that is about to write
  into a block whose count is above one gets a newly taken block, the shared block
  is copied into it, and the shared block's count drops by one; the last holder
  then writes in place.
* vLLM-SOSP23 note, "core method": fork / append / free are the primitives that
  parallel sampling, beam search and shared prefixes are built from.
* vLLM post, "3. scheduling and preemption", swapping: eviction is all-or-nothing per
  request (all of its blocks move together) to CPU memory, whose blocks a CPU block
  allocator manages; when the request resumes its blocks are copied back. Here a
  swap of several requests maps each distinct device block they name to one host
  block (so blocks they share stay shared), returns the (from, to) copies, moves the
  references from one pool to the other and frees blocks left without any.

Readings where the pages are silent: the free pool hands out blocks first in, first
out, in an order the caller may give (default 0, 1, 2, ...), and freed blocks join
its back in table order; a request's append either completes or, when the pool has
too few free blocks, changes nothing; positions are written in increasing order, so
only a sequence's last (partially filled) block can need a copy. The host pool
follows the same rules; a request swapped out can be swapped in or freed, nothing
else; a swap takes blocks in the order the listed requests' tables name them.
"""
from collections import deque


class OutOfBlocks(RuntimeError):
    pass


class BlockManager:
    """Host-side bookkeeping of one KV block pool.

    ``mutation`` != 0 plants a deliberate mistake (used only by the test that
    checks that the pins catch it): 1 copy-on-write keeps the shared block's count,
    2 shared blocks are written in place, 3 the offset in the block is off by one,
    4 freed blocks are not returned, 5 fork does not count the child's references,
    6 a swap copies a shared block once per reference, 7 a swap keeps the references
    in the pool it leaves.
    """

    def __init__(self, num_blocks: int, block_size: int, free_order=None, mutation: int = 0,
                 num_host_blocks: int = 0, host_free_order=None):
        if num_blocks <= 0 or block_size <= 0 or num_host_blocks < 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must list every block once")
        horder = (list(range(num_host_blocks)) if host_free_order is None
                  else [int(b) for b in host_free_order])
        if sorted(horder) != list(range(num_host_blocks)):
            raise ValueError("host_free_order must list every host block once")
        self.B = block_size
        self.num_blocks = num_blocks
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.hfree = deque(horder)
        self.href = [0] * num_host_blocks
        self.tables = {}     # sequence id -> physical block ids of its logical blocks
        self.lens = {}       # sequence id -> tokens held
        self.on_host = set() # sequences whose blocks are in the host pool
        self.mutation = mutation

    def _on_device(self, seq):
        if seq not in self.tables:
            raise KeyError(f"unknown sequence {seq}")
        if seq in self.on_host:
            raise KeyError(f"sequence {seq} is swapped out")

    # ---- primitives
    def add(self, seq) -> None:
        """A new request with no tokens yet."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq} exists")
        self.tables[seq] = []
        self.lens[seq] = 0

    def fork(self, parent, child) -> None:
        """The child shares every block of the parent (each count + 1)."""
        if parent not in self.tables or child in self.tables:
            raise KeyError("fork needs an existing parent and a new child")
        self._on_device(parent)
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        if self.mutation != 5:
            for b in self.tables[child]:
                self.ref[b] += 1

    def free_seq(self, seq) -> None:
        """A finished request: each of its blocks loses one reference; blocks left with
        none return to the pool."""
        if seq in self.on_host:
            self.on_host.discard(seq)
            ref, free = self.href, self.hfree
        else:
            ref, free = self.ref, self.free
        for b in self.tables.pop(seq):
            ref[b] -= 1
            if ref[b] == 0 and self.mutation != 4:
                free.append(b)
        del self.lens[seq]

    def _blocks_needed(self, seq, n, shared_left) -> int:
        """Free blocks one append of n tokens takes, given the counts the earlier
        appends of the same batch leave (shared_left: block -> count)."""
        L, B = self.lens[seq], self.B
        table = self.tables[seq]
        need = 0
        if n <= 0:
            return 0
        if L % B != 0:
            last = table[-1]
            if shared_left.get(last, self.ref[last]) > 1:
                need += 1
                shared_left[last] = shared_left.get(last, self.ref[last]) - 1
        need += -(-(L + n) // B) - len(table)
        return need

    def append(self, seq, n: int):
        """Reserve slots for n new tokens at positions L .. L + n - 1.

        Returns (slots, copies): slot of each new token (block * B + offset) and the
        (source, destination) block copies the write needs first."""
        return self.append_batch([seq], [n])

    def append_batch(self, seqs, ns):
        """One step: the new tokens of several requests, in the order given (the first
        writer into a shared block copies it). All-or-nothing on pool exhaustion."""
        if len(seqs) != len(ns):
            raise ValueError("one count per sequence")
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence appears twice in one step")
        for s, n in zip(seqs, ns):
            self._on_device(s)
            if n < 0:
                raise ValueError("negative token count")
        shared_left = {}
        need = sum(self._blocks_needed(s, n, shared_left) for s, n in zip(seqs, ns))
        if need > len(self.free):
            raise OutOfBlocks(f"{need} blocks needed, {len(self.free)} free")
        slots, copies = [], []
        B = self.B
        for s, n in zip(seqs, ns):
            table = self.tables[s]
            for p in range(self.lens[s], self.lens[s] + n):
                j = p // B
                if j == len(table):
                    b = self.free.popleft()
                    self.ref[b] = 1
                    table.append(b)
                elif self.ref[table[j]] > 1 and self.mutation != 2:
                    old = table[j]
                    b = self.free.popleft()
                    self.ref[b] = 1
                    if self.mutation != 1:
                        self.ref[old] -= 1
                    copies.append((old, b))
                    table[j] = b
                off = (p - 1) % B if self.mutation == 3 else p % B
                slots.append(table[j] * B + off)
            self.lens[s] += n
        return slots, copies

    def _swap(self, seqs, out: bool):
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence appears twice in one swap")
        for q in seqs:
            if q not in self.tables:
                raise KeyError(f"unknown sequence {q}")
            if (q in self.on_host) == out:
                raise KeyError(f"sequence {q} is already {'out' if out else 'in'}")
        src_ref, src_free = (self.ref, self.free) if out else (self.href, self.hfree)
        dst_ref, dst_free = (self.href, self.hfree) if out else (self.ref, self.free)
        distinct = []
        for q in seqs:
            for b in self.tables[q]:
                if b not in distinct or self.mutation == 6:
                    distinct.append(b)
        if len(distinct) > len(dst_free):
            raise OutOfBlocks(f"{len(distinct)} blocks needed, {len(dst_free)} free")
        to = {}
        pairs = []
        for b in distinct:
            c = dst_free.popleft()
            to[b] = c
            pairs.append((b, c))
        for q in seqs:
            t = self.tables[q]
            for j, b in enumerate(t):
                dst_ref[to[b]] += 1
                if self.mutation != 7:
                    src_ref[b] -= 1
                    if src_ref[b] == 0:
                        src_free.append(b)
                t[j] = to[b]
            if out:
                self.on_host.add(q)
            else:
                self.on_host.discard(q)
        return pairs

    def swap_out(self, seqs):
        """All blocks of the listed requests go to the host pool; returns the
        (device block, host block) copies to make before the device blocks are reused."""
        return self._swap(list(seqs), True)

    def swap_in(self, seqs):
        """The listed swapped-out requests come back; returns the (host block, device
        block) copies to make before they run."""
        return self._swap(list(seqs), False)

    # ---- views
    def table(self, seq):
        return list(self.tables[seq])

    def filled(self, seq) -> int:
        """#filled of the request's last block (0 for a request without blocks)."""
        L = self.lens[seq]
        return 0 if L == 0 else L - self.B * (-(-L // self.B) - 1)

    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def host_refcount(self, block: int) -> int:
        return self.href[block]

    def num_free_host(self) -> int:
        return len(self.hfree)

    def is_on_host(self, seq) -> bool:
        if seq not in self.tables:
            raise KeyError(f"unknown sequence {seq}")
        return seq in self.on_host
