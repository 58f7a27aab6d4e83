"""The decode scorer's mbarrier protocol (index_decode_mx_kernel), checked on the CPU.

A model of the kernel's roles under random interleavings. The ring size is read from the
kernel source, so that the model follows the kernel.
- The producer's copies fill stage u mod kMSlots with unit u's code rows once the MMAs of unit
  u - kMSlots have completed (done). A copy lands some time after it is issued (s_full).
- Four scale warps write unit u's scale words into TMEM slot u mod kMSlots once the epilogue
  has read that slot's accumulators (d_free), then wait for the unit's codes (s_full) and
  release the unit to the MMA thread (sf_full).
- Two MMA threads issue the even / odd units' MMAs after sf_full; each thread's MMAs complete
  asynchronously and in its issue order (done).
- Eight epilogue warps read every unit's accumulators in order and free them (d_free).

Barrier semantics are those of `mbarrier.try_wait.parity`: a wait for parity P succeeds once
the barrier's number of completed phases has the other parity.

At every hand-off the model asserts that the consumer sees the intended unit:
- a copy lands in a stage only after the MMAs that read the stage's previous unit completed;
- scale words are overwritten only after the MMAs that read them completed;
- an MMA reads its own unit's codes and scale words, and writes accumulators the epilogue
  has already read;
- the epilogue reads its own unit's scores.

It also asserts that every epilogue warp reaches the last unit (no deadlock). A second test
removes each wait in turn and checks that the model then reports a violation.
"""
import random
import re
from pathlib import Path

SRC = Path(__file__).resolve().parent.parent / "compressed_sparse_attention_03_gb300" / "csrc" / "csa2_index_tc.cu"
TEXT = SRC.read_text()


def _const(name: str) -> int:
    m = re.search(rf"\b{name}\s*=\s*(\d+)", TEXT)
    assert m, f"{name} not found in {SRC.name}"
    return int(m.group(1))


SLOTS = _const("kMSlots")
SF_WARPS, EPI_WARPS = 4, 8


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def ready(self, parity):
        return (self.completed & 1) != parity


def prev_ready(bar, u):
    """The wait of unit u on the slot's previous use (none for the first kMSlots units)."""
    return u < SLOTS or bar.ready(((u // SLOTS) - 1) & 1)


def simulate(nu: int, seed: int, skip: str = "") -> None:
    rng = random.Random(seed)
    s_full = [Bar(1) for _ in range(SLOTS)]
    sf_full = [Bar(SF_WARPS) for _ in range(SLOTS)]
    done = [Bar(1) for _ in range(SLOTS)]
    d_free = [Bar(EPI_WARPS) for _ in range(SLOTS)]
    stage = [None] * SLOTS                          # unit whose codes the stage holds
    sfw = [[None] * SF_WARPS for _ in range(SLOTS)]  # unit whose scale words each quarter holds
    acc = [None] * SLOTS                            # unit whose scores the accumulators hold
    prod, copies = 0, []
    sf = [{"u": 0, "written": False} for _ in range(SF_WARPS)]
    mma, inflight = [0, 1], []  # next unit of each MMA thread; (thread, unit) in flight
    epi = [0] * EPI_WARPS
    mma_done, epi_read = set(), set()
    while True:
        acts = []
        if prod < nu and (skip == "prod_done" or prev_ready(done[prod % SLOTS], prod)):
            acts.append(("prod", 0))
        if copies:
            acts.append(("land", 0))
        for w, d in enumerate(sf):
            u = d["u"]
            if u >= nu:
                continue
            if not d["written"] and (skip == "sf_dfree" or prev_ready(d_free[u % SLOTS], u)):
                acts.append(("sf_write", w))
            elif d["written"] and (skip == "sf_sfull" or s_full[u % SLOTS].ready((u // SLOTS) & 1)):
                acts.append(("sf_release", w))
        for e in (0, 1):
            u = mma[e]
            if u < nu and sf_full[u % SLOTS].ready((u // SLOTS) & 1):
                acts.append(("issue", e))
        if inflight:
            acts.append(("complete", rng.choice(sorted({e for e, _ in inflight}))))
        for w, u in enumerate(epi):
            if u < nu and (skip == "epi_done" or done[u % SLOTS].ready((u // SLOTS) & 1)):
                acts.append(("epi", w))
        if not acts:
            break
        kind, who = rng.choice(acts)
        if kind == "prod":
            copies.append(prod)
            prod += 1
        elif kind == "land":
            u = copies.pop(rng.randrange(len(copies)))
            s = u % SLOTS
            assert stage[s] in (None, u - SLOTS), f"stage {s}: unit {stage[s]} then {u}"
            assert stage[s] is None or stage[s] in mma_done, f"stage {s} overwritten before unit {stage[s]}'s MMAs"
            stage[s] = u
            s_full[s].arrive()
        elif kind == "sf_write":
            d = sf[who]
            u, s = d["u"], d["u"] % SLOTS
            prev = sfw[s][who]
            assert prev in (None, u - SLOTS), f"scale slot {s}: unit {prev} then {u}"
            assert prev is None or prev in mma_done, f"scale slot {s} overwritten before unit {prev}'s MMAs"
            sfw[s][who] = u
            d["written"] = True
        elif kind == "sf_release":
            d = sf[who]
            sf_full[d["u"] % SLOTS].arrive()
            d["u"] += 1
            d["written"] = False
        elif kind == "issue":
            u = mma[who]
            s = u % SLOTS
            assert stage[s] == u, f"MMA of unit {u}: stage holds {stage[s]}"
            assert all(x == u for x in sfw[s]), f"MMA of unit {u}: scale slot holds {sfw[s]}"
            assert u < SLOTS or (u - SLOTS) in epi_read, f"accumulators {s} reused before unit {u - SLOTS} was read"
            inflight.append((who, u))
            mma[who] += 2
        elif kind == "complete":
            k = next(n for n, (e, _) in enumerate(inflight) if e == who)
            _, u = inflight.pop(k)
            s = u % SLOTS
            assert stage[s] == u and all(x == u for x in sfw[s]), f"MMA of unit {u} saw its operands change"
            acc[s] = u
            mma_done.add(u)
            done[s].arrive()
        elif kind == "epi":
            u = epi[who]
            assert acc[u % SLOTS] == u, f"epilogue of unit {u}: accumulators hold unit {acc[u % SLOTS]}"
            d_free[u % SLOTS].arrive()
            epi[who] += 1
            if all(x > u for x in epi):
                epi_read.add(u)
    assert epi == [nu] * EPI_WARPS, f"stopped at {epi} of {nu} units (deadlock)"
    assert not inflight and not copies


def test_slots_keep_their_mma_thread():
    assert SLOTS % 2 == 0
    assert re.search(r"for \(int u = warp - kMMma; u < nu; u \+= 2\)", TEXT)


def test_barrier_counts_match_the_roles():
    assert re.search(r"mbar_init\(&bars\.sf_full\[i\],\s*4\)", TEXT)
    assert re.search(r"mbar_init\(&bars\.d_free\[i\],\s*8\)", TEXT)
    assert re.search(r"mbar_init\(&bars\.done\[i\],\s*1\)", TEXT)


def test_random_interleavings():
    for nu in (1, 2, 3, 5, 6, 7, 12, 13, 108, 109):
        for seed in range(40 if nu < 100 else 8):
            simulate(nu, 1000 * nu + seed)


def test_each_wait_is_needed():
    # without any one of the waits, some interleaving breaks a hand-off
    for skip in ("prod_done", "sf_dfree", "sf_sfull", "epi_done"):
        caught = False
        for seed in range(400):
            try:
                simulate(13, seed, skip)
            except AssertionError:
                caught = True
                break
        assert caught, f"the model did not notice the missing wait {skip}"
