"""The decode scorer's mbarrier protocol (index_decode_tc_kernel), checked on the CPU.

A model of the kernel's roles under random interleavings. The pipeline constants are read
from the kernel source, so that the model follows the kernel.
- The producer fills a ring of code stages, each holding a pair of key tiles.
- Four decoder groups take tiles i = group mod 4 into TMEM A slots (i mod kDSlots), and give
  a tile's stage back to the producer when they mark its slot full.
- Two MMA issuers take even and odd tiles into accumulators i mod 4. Each issuer's MMAs
  complete asynchronously and in order.
- The epilogue reads every accumulator in tile order.

Barrier semantics are those of `mbarrier.try_wait.parity`: a wait for parity P succeeds once
the barrier's number of completed phases has the other parity.

At every hand-off the model asserts that the consumer sees the intended tile:
- a stage holds the decoders' group;
- a slot is overwritten only after its previous tile's MMAs completed;
- an MMA reads its own tile;
- an accumulator is reused only after the epilogue read it.

It also asserts that the epilogue reaches the last tile (no deadlock). Tile counts include
odd ones and a last tile of one key, as on a 524,289-entry row.
"""
import random
import re
from pathlib import Path

SRC = Path(__file__).resolve().parent.parent / "compressed_sparse_attention_03_gb300" / "csrc" / "csa2_index_tc.cu"


def _const(name: str) -> int:
    m = re.search(rf"\b{name}\s*=\s*(\d+)", SRC.read_text())
    assert m, f"{name} not found in {SRC.name}"
    return int(m.group(1))


SLOTS, ACC, GROUPS = _const("kDSlots"), _const("kDAcc"), _const("kDGroups")
GROUP, STAGES = _const("kDGroup"), _const("kDStages")
WARPS_PER_GROUP = 4  # a decoder group and the epilogue are four warps (one per TMEM lane quarter)


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


def simulate(nt: int, seed: int) -> None:
    rng = random.Random(seed)
    s_full = [Bar(1) for _ in range(STAGES)]
    s_empty = [Bar(WARPS_PER_GROUP * GROUP) for _ in range(STAGES)]
    a_full = [Bar(WARPS_PER_GROUP) for _ in range(SLOTS)]
    done = [Bar(1) for _ in range(SLOTS)]
    d_free = [Bar(WARPS_PER_GROUP) for _ in range(ACC)]
    stage, slot, acc = [None] * STAGES, [None] * SLOTS, [None] * ACC
    ng = (nt + GROUP - 1) // GROUP
    prod = 0
    dec = [{"g": w // WARPS_PER_GROUP, "i": w // WARPS_PER_GROUP, "read": False}
           for w in range(GROUPS * WARPS_PER_GROUP)]
    iss = [0, 1]  # next tile of each issuer (even / odd tiles)
    epi = [0] * WARPS_PER_GROUP
    inflight = []  # (issuer, tile)
    mma_done, epi_read = set(), set()
    while True:
        acts = []
        if prod < ng and (prod < STAGES or s_empty[prod % STAGES].ready(((prod // STAGES) - 1) & 1)):
            acts.append(("prod", 0))
        for w, d in enumerate(dec):
            i = d["i"]
            if i >= nt:
                continue
            gi = i // GROUP
            if not d["read"] and s_full[gi % STAGES].ready((gi // STAGES) & 1):
                acts.append(("dec_read", w))
            elif d["read"] and (i < SLOTS or done[i % SLOTS].ready(((i // SLOTS) - 1) & 1)):
                acts.append(("dec_write", w))
        for e, i in enumerate(iss):
            if i < nt and a_full[i % SLOTS].ready((i // SLOTS) & 1) and (
                    i < ACC or d_free[i % ACC].ready(((i // ACC) - 1) & 1)):
                acts.append(("issue", e))
        if inflight:
            acts.append(("complete", rng.choice(sorted({e for e, _ in inflight}))))
        for w, i in enumerate(epi):
            if i < nt and done[i % SLOTS].ready((i // SLOTS) & 1):
                acts.append(("epi", w))
        if not acts:
            break
        kind, who = rng.choice(acts)
        if kind == "prod":
            stage[prod % STAGES] = prod
            s_full[prod % STAGES].arrive()
            prod += 1
        elif kind == "dec_read":
            d = dec[who]
            s = (d["i"] // GROUP) % STAGES
            assert stage[s] == d["i"] // GROUP, f"tile {d['i']}: stage {s} holds group {stage[s]}"
            d["read"] = True
        elif kind == "dec_write":
            d = dec[who]
            i, sl = d["i"], d["i"] % SLOTS
            prev = slot[sl]
            assert prev in (None, i, i - SLOTS), f"slot {sl}: tile {prev} then {i}"
            assert prev in (None, i) or prev in mma_done, f"slot {sl} rewritten before tile {prev}'s MMAs completed"
            slot[sl] = i
            # the stage is released with the slot (after the TMEM store and a proxy fence)
            s_empty[(i // GROUP) % STAGES].arrive()
            a_full[sl].arrive()
            d["read"] = False
            d["i"] += GROUPS
        elif kind == "issue":
            i = iss[who]
            assert slot[i % SLOTS] == i, f"MMA of tile {i}: slot holds {slot[i % SLOTS]}"
            assert i < ACC or (i - ACC) in epi_read, f"accumulator {i % ACC} reused before tile {i - ACC} was read"
            inflight.append((who, i))
            iss[who] += 2
        elif kind == "complete":
            k = next(n for n, (e, _) in enumerate(inflight) if e == who)
            _, i = inflight.pop(k)
            assert slot[i % SLOTS] == i, f"MMA of tile {i} completed reading tile {slot[i % SLOTS]}"
            acc[i % ACC] = i
            mma_done.add(i)
            done[i % SLOTS].arrive()
        elif kind == "epi":
            i = epi[who]
            assert acc[i % ACC] == i, f"epilogue of tile {i}: accumulator holds tile {acc[i % ACC]}"
            d_free[i % ACC].arrive()
            epi[who] += 1
            if all(x > i for x in epi):
                epi_read.add(i)
    assert epi == [nt] * WARPS_PER_GROUP, f"stopped at {epi} of {nt} tiles (deadlock)"
    assert not inflight


def test_constants_keep_each_slot_and_accumulator_with_one_issuer():
    assert SLOTS % 2 == 0 and ACC % 2 == 0
    assert GROUP == 2


def test_random_interleavings():
    for nt in (1, 2, 3, 4, 5, 6, 7, 11, 13, 26, 208, 209):
        for seed in range(40 if nt < 100 else 8):
            simulate(nt, 1000 * nt + seed)
