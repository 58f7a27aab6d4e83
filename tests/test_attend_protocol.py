"""The attention kernel's synchronisation protocol (attend_tc_kernel, one query), checked on
the CPU: a model of its 14 warps under random interleavings.

Roles, as in the kernel:
- **Producer warps 4-11.** Each converts its share of Q and arrives on q_full, then meets the
  other producers on named barrier 2. Per chunk it refills the four 128-dim tiles of G (two
  atoms each) once tile_free says the last chunk's O MMAs have read them.
- **Producer warps 4-7 also** take heads 32-63 of each chunk's softmax.
- **Softmax warps 0-3** take heads 0-31, and alone run the rare "new reference" path (O and
  the row sums rescaled in TMEM).
- **Two MMA threads.** The S thread issues S over the eight atoms as they fill and commits to
  s_full (the atoms are refilled only after the last chunk's O MMAs, which follow p_full, so S
  is overwritten only after every warp read it). The O thread issues the
  four O tiles and the row sums after p_full, with commits to tile_free[m] and l_done. Each
  thread's MMAs run asynchronously and in its own issue order; the two streams interleave in
  any order, and a commit covers only its own thread's MMAs.
- **Softmax and helpers** wait for l_done of the last chunk before they rewrite P.
- **Warps 0-11** meet on named barrier 3 and read O.

mbarriers follow `mbarrier.try_wait.parity` semantics. Named barriers follow `bar.sync`:
arrivals count toward the barrier's current generation, whichever phase the arriving warp
means.

At every hand-off the model asserts the data it sees:
- atoms are rewritten only after the MMAs that read the last chunk completed;
- MMAs read the intended chunk's atoms and P;
- the S accumulator is read for its own chunk, and overwritten only after every warp read it;
- P is rewritten only after the last chunk's O and row-sum MMAs read it;
- O is rescaled only between chunks;
- the softmax references are read only when no warp is writing them;
- the output is read after the last MMA.

It also asserts that every warp finishes (no deadlock) and that no barrier generation mixes
phases.

The model orders events; it does not model memory visibility. Barrier 5, for producer warps
4-7, is therefore redundant here and planting its removal is not caught: it makes the softmax
warps' reference updates visible to the helpers, which also reach a chunk only after p_full of
the last chunk. The l_done waits before P is rewritten are taken by both the softmax warps and
the helpers, and barrier 5 joins them, so only the removal of both is caught. A skipped
tile_free wait, a p_full count without the helpers, and an early read of the references are
caught too.
"""
import random

NQ = 4  # softmax warps; producer warps 4-7 are the helpers


class MBar:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity):
        return (self.completed & 1) != parity


class NBar:
    def __init__(self, nwarps):
        self.n, self.arrived, self.gen, self.tags = nwarps, 0, 0, set()

    def arrive(self, tag):
        self.tags.add(tag)
        self.arrived += 1
        g = self.gen
        if self.arrived == self.n:
            assert len(self.tags) == 1, f"one barrier generation mixed phases {sorted(self.tags)}"
            self.gen, self.arrived, self.tags = self.gen + 1, 0, set()
        return g


class Model:
    def __init__(self, nloc, redo, rng):
        self.nloc, self.redo, self.rng = nloc, redo, rng
        self.q_full, self.s_full, self.p_full, self.l_done = MBar(8), MBar(1), MBar(8), MBar(1)
        self.atom_full = [MBar(8) for _ in range(8)]
        self.tile_free = [MBar(1) for _ in range(4)]
        self.nbar = {1: NBar(4), 2: NBar(8), 3: NBar(12), 4: NBar(8), 5: NBar(8)}
        self.atom_writes = {}          # (atom, chunk) -> warps that wrote their rows
        self.atom_chunk = [None] * 8   # newest chunk written into an atom
        self.p_writes = {}             # (half, chunk) -> warp writes
        self.p_chunk = [None, None]
        self.s_acc = None              # chunk whose S is in TMEM
        self.s_reads = {}              # chunk -> warps that read S
        self.s_mmas = {}               # chunk -> S MMAs completed
        self.done = set()              # completed MMAs: ("S", i, k), ("O", i, m), ("L", i)
        self.o_chunk = [None] * 4
        self.l_chunk = None
        self.issued_o = set()          # chunks whose O MMAs were issued
        self.red_max = {}              # (chunk, half) -> writes
        self.m_ref_writers = 0         # warps inside the reference-writing window
        self.queues = {"S": [], "O": []}  # each MMA thread's async operations, in its order

    # -- helpers
    def nsync(self, bid, tag):
        g = self.nbar[bid].arrive(tag)
        yield lambda: self.nbar[bid].gen > g

    def write_atom(self, k, i):
        if i > 0:
            assert ("S", i - 1, k) in self.done, f"atom {k} rewritten before S of chunk {i-1} read it"
            assert ("O", i - 1, k // 2) in self.done, f"atom {k} rewritten before O tile {k//2} of chunk {i-1} read it"
        self.atom_writes[(k, i)] = self.atom_writes.get((k, i), 0) + 1
        self.atom_chunk[k] = i

    def write_p(self, half, i):
        if i > 0:
            assert all(("O", i - 1, m) in self.done for m in range(4)) and ("L", i - 1) in self.done, \
                f"P half {half} of chunk {i} written before the last chunk's O / row-sum MMAs read P"
        assert i not in self.issued_o, f"P of chunk {i} written after its O MMAs were issued"
        self.p_writes[(half, i)] = self.p_writes.get((half, i), 0) + 1
        self.p_chunk[half] = i

    def read_s(self, i, w):
        assert self.s_acc == i and self.s_mmas.get(i) == 8, f"warp {w} read S of chunk {self.s_acc} for chunk {i}"
        self.s_reads[i] = self.s_reads.get(i, 0) + 1

    def read_m_ref(self):
        assert self.m_ref_writers == 0, "references read while being written"

    # -- roles
    def producer(self, w):  # w = 0..7 for warps 4..11
        helper = w < 4
        if self.nloc > 0:
            self.q_full.arrive()
            yield from self.nsync(2, "q")
        for i in range(self.nloc):
            for at in range(4):
                if i > 0:
                    yield lambda at=at, i=i: self.tile_free[at].ready((i - 1) & 1)
                for k in (2 * at, 2 * at + 1):
                    self.write_atom(k, i)
                self.atom_full[2 * at].arrive()
                self.atom_full[2 * at + 1].arrive()
            if helper:
                yield lambda i=i: self.s_full.ready(i & 1)
                if i > 0:
                    yield lambda i=i: self.l_done.ready((i - 1) & 1)
                self.read_s(i, 4 + w)
                if i == 0:
                    self.red_max[(0, 1)] = self.red_max.get((0, 1), 0) + 1
                    yield from self.nsync(5, ("c", i))
                    yield from self.nsync(4, ("r", i))
                    self.read_m_ref()
                    self.write_p(1, i)
                else:
                    yield from self.nsync(5, ("c", i))
                    self.read_m_ref()
                    self.write_p(1, i)
                    yield from self.nsync(4, ("r", i))
                self.p_full.arrive()
        yield from self.nsync(3, "out")
        self.read_output()

    def softmax(self, w):
        for i in range(self.nloc):
            yield lambda i=i: self.s_full.ready(i & 1)
            if i > 0:
                yield lambda i=i: self.l_done.ready((i - 1) & 1)
            self.read_s(i, w)
            if i == 0:
                self.red_max[(0, 0)] = self.red_max.get((0, 0), 0) + 1
                yield from self.nsync(5, ("c", i))
                if w < 2:  # threads 0..63 set the references (a window other warps may interleave with)
                    assert self.red_max.get((0, 0)) == NQ and self.red_max.get((0, 1)) == NQ, "chunk maxima incomplete"
                    self.m_ref_writers += 1
                    yield lambda: True
                    self.m_ref_writers -= 1
                yield from self.nsync(4, ("r", i))
                self.read_m_ref()
                self.write_p(0, i)
            else:
                yield from self.nsync(5, ("c", i))
                self.read_m_ref()
                self.write_p(0, i)
                yield from self.nsync(4, ("r", i))
                if self.redo[i]:
                    self.red_max[(i, 0)] = self.red_max.get((i, 0), 0) + 1
                    yield from self.nsync(1, ("m1", i))
                    if w < 2:
                        assert self.red_max.get((i, 0)) == NQ
                        self.m_ref_writers += 1
                        yield lambda: True
                        self.m_ref_writers -= 1
                    yield from self.nsync(1, ("m2", i))
                    yield lambda i=i: self.l_done.ready((i - 1) & 1)
                    assert all(self.o_chunk[m] == i - 1 for m in range(4)) and self.l_chunk == i - 1, \
                        "O rescaled while MMAs of another chunk are pending"
                    assert i not in self.issued_o
                    self.write_p(0, i)
                    self.write_p(1, i)
            self.p_full.arrive()
        if self.nloc > 0:
            yield lambda: self.l_done.ready((self.nloc - 1) & 1)
        yield from self.nsync(3, "out")
        self.read_output()

    def issuer_s(self):
        if self.nloc == 0:
            return
        q = self.queues["S"]
        yield lambda: self.q_full.ready(0)
        for i in range(self.nloc):
            for k2 in range(4):
                yield lambda k2=k2, i=i: self.atom_full[2 * k2].ready(i & 1) and self.atom_full[2 * k2 + 1].ready(i & 1)
                for k in (2 * k2, 2 * k2 + 1):
                    assert self.atom_writes.get((k, i)) == 8, f"S of chunk {i} issued on atom {k} not fully written"
                    q.append(("S", i, k))
            q.append(("commit", self.s_full))

    def issuer_o(self):
        if self.nloc == 0:
            return
        q = self.queues["O"]
        for i in range(self.nloc):
            yield lambda i=i: self.p_full.ready(i & 1)
            assert self.s_reads.get(i) == 8, "O issued before every warp read S"
            self.issued_o.add(i)
            for m in range(4):
                q.append(("O", i, m))
                q.append(("commit", self.tile_free[m]))
            q.append(("L", i))
            q.append(("commit", self.l_done))

    def tensor_step(self, which):
        op = self.queues[which].pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, i = op[0], op[1]
        if kind == "S":
            k = op[2]
            assert self.atom_chunk[k] == i, f"S of chunk {i} read atom {k} holding chunk {self.atom_chunk[k]}"
            if self.s_acc != i:
                assert i == 0 or self.s_reads.get(i - 1) == 8, f"S of chunk {i} overwrote S before chunk {i-1} was read"
                self.s_acc, self.s_mmas[i] = i, 0
            self.s_mmas[i] += 1
            self.done.add(("S", i, k))
        elif kind == "O":
            m = op[2]
            for k in (2 * m, 2 * m + 1):
                assert self.atom_chunk[k] == i, f"O tile {m} of chunk {i} read atom {k} holding {self.atom_chunk[k]}"
            assert self.p_chunk == [i, i], f"O of chunk {i} read P of chunks {self.p_chunk}"
            self.o_chunk[m] = i
            self.done.add(("O", i, m))
        else:
            assert self.p_chunk == [i, i]
            self.l_chunk = i
            self.done.add(("L", i))

    def read_output(self):
        if self.nloc:
            last = self.nloc - 1
            assert all(("O", last, m) in self.done for m in range(4)) and ("L", last) in self.done, \
                "output read before the last MMAs completed"


def simulate(nloc, seed):
    rng = random.Random(seed)
    redo = [False] + [rng.random() < 0.3 for _ in range(1, max(nloc, 1))]
    md = Model(nloc, redo, rng)
    pace = rng.choice([0.02, 0.1, 0.3, 0.6])
    agents = [md.softmax(w) for w in range(NQ)] + [md.producer(w) for w in range(8)] + [md.issuer_s(), md.issuer_o()]
    waits = [None] * len(agents)
    live = list(range(len(agents)))

    def advance(a):
        try:
            waits[a] = next(agents[a])
        except StopIteration:
            waits[a] = "end"

    for a in list(live):
        advance(a)
    while True:
        ready = [a for a in range(len(agents)) if waits[a] != "end" and waits[a]()]
        tensor = [("tensor", k) for k in md.queues if md.queues[k]]
        agent = [("agent", a) for a in ready]
        if not tensor and not agent:
            break
        # the tensor pipe's pace relative to the warps varies per run (slow MMAs open the races)
        kind, a = rng.choice(tensor if tensor and (not agent or rng.random() < pace) else agent)
        if kind == "tensor":
            md.tensor_step(a)
        else:
            advance(a)
    stuck = [a for a in range(len(agents)) if waits[a] != "end"]
    assert not stuck, f"nloc={nloc}: warps {stuck} never finished (deadlock)"
    assert not md.queues["S"] and not md.queues["O"]


def test_random_interleavings():
    for nloc in (0, 1, 2, 3, 5):
        for seed in range(60 if nloc < 2 else 300):
            simulate(nloc, 1000 * nloc + seed)
