"""A discrete-event model of the one-SM tensor-core kernel's barrier protocol.

The kernel (tc_gemm.cu) runs three rings between a TMA producer thread, an
MMA thread and `groups` groups of four dequantizing warps, handing stages over
with mbarriers whose waits test only the parity of a phase. A parity wait
names its phase correctly only while the barrier is at most one phase away
from it; the ring depths have to guarantee that. This model replays the
protocol step by step under random interleavings and random copy and MMA
latencies, with barriers that behave as the hardware's (a phase completes
after `count` arrivals; a wait for parity P passes when the completed-phase
count's parity differs from P), and checks every wait that passes against
what it is meant to prove: the stage's codes or activations have landed, the
MMAs that read a tensor-memory slot have completed, a slot is not refilled
before its last use, and no barrier phase mixes arrivals of two stages.

Per stage the roles do what the kernel does, in its order:
  producer      polls code_empty / stage_done of its next copy of each ring
                (the first ring of codes may go out before anything else);
  MMA thread    waits dq_full of the next stage, issues its MMAs, commits to
                stage_done (MMAs complete in issue order, after a delay);
  dequant warp  waits code_full; with more atoms per stage than it converts
                at once, waits for its tensor-memory slot first; reads the
                codes and arrives on code_empty; otherwise waits for its slot
                now; converts; waits act_full; arrives on dq_full.
"""
from __future__ import annotations

import random


class Barrier:
    def __init__(self, count: int, name: str):
        self.count, self.pending, self.completed, self.name = count, count, 0, name
        self.tags: list = []

    def arrive(self, tag) -> None:
        self.tags.append(tag)
        self.pending -= 1
        if self.pending == 0:
            if len(set(self.tags)) != 1:
                raise AssertionError(f"{self.name}: one phase mixes arrivals {self.tags}")
            self.tags = []
            self.completed += 1
            self.pending = self.count

    def passes(self, parity: int) -> bool:
        return (self.completed & 1) != parity


def simulate(nk: int, code_slots: int, act_slots: int, dq_slots: int, groups: int,
             seed: int, slot_first: bool = False, early_codes: bool = True,
             max_steps: int = 200_000) -> str:
    """One random run of `nk` stages. Returns "ok", or raises AssertionError
    (a wait passed on the wrong phase, or a slot was reused too early), or
    returns "deadlock ..." if no role can move."""
    rnd = random.Random(seed)
    code_full = [Barrier(1, f"code_full[{i}]") for i in range(code_slots)]
    code_empty = [Barrier(4, f"code_empty[{i}]") for i in range(code_slots)]
    act_full = [Barrier(1, f"act_full[{i}]") for i in range(act_slots)]
    stage_done = [Barrier(1, f"stage_done[{i}]") for i in range(act_slots)]
    dq_full = [Barrier(4, f"dq_full[{i}]") for i in range(dq_slots)]
    now = 0
    events: list = []
    codes_landed, acts_landed, consumed, mma_done, converted = set(), set(), set(), set(), set()

    def later(delay, fn):
        events.append((now + delay, len(events), fn))

    def copy_codes(kb):
        def land():
            codes_landed.add(kb)
            code_full[kb % code_slots].arrive(("codes", kb))
        later(rnd.randint(1, 40), land)

    def copy_acts(kb):
        def land():
            acts_landed.add(kb)
            act_full[kb % act_slots].arrive(("acts", kb))
        later(rnd.randint(1, 40), land)

    prod = {"ci": 0, "ai": 0}
    if early_codes:
        while prod["ci"] < min(nk, code_slots):
            copy_codes(prod["ci"])
            prod["ci"] += 1

    def producer() -> bool:
        moved = False
        ci, ai = prod["ci"], prod["ai"]
        if ci < nk and code_empty[ci % code_slots].passes(((ci // code_slots) & 1) ^ 1):
            if ci >= code_slots and (ci - code_slots) not in consumed:
                raise AssertionError(f"code slot of stage {ci} refilled before stage "
                                     f"{ci - code_slots} read it")
            copy_codes(ci)
            prod["ci"] += 1
            moved = True
        if ai < nk and stage_done[ai % act_slots].passes(((ai // act_slots) & 1) ^ 1):
            if ai >= act_slots and (ai - act_slots) not in mma_done:
                raise AssertionError(f"activation slot of stage {ai} refilled before the "
                                     f"MMAs of stage {ai - act_slots} completed")
            copy_acts(ai)
            prod["ai"] += 1
            moved = True
        return moved

    mma = {"kb": 0, "busy_until": 0}

    def mma_thread() -> bool:
        kb = mma["kb"]
        if kb >= nk or not dq_full[kb % dq_slots].passes((kb // dq_slots) & 1):
            return False
        if kb not in converted or kb not in acts_landed:
            raise AssertionError(f"MMAs of stage {kb} issued before its operands were ready")
        mma["kb"] += 1
        done_at = max(now, mma["busy_until"]) + rnd.randint(1, 30)   # in issue order
        mma["busy_until"] = done_at

        def complete(kb=kb):
            mma_done.add(kb)
            stage_done[kb % act_slots].arrive(("mma", kb))
        events.append((done_at, len(events), complete))
        return True

    warps = [{"g": g, "kb": g, "step": 0} for g in range(groups) for _ in range(4)]

    def slot_ready(kb) -> bool:
        if kb < dq_slots:
            return True
        prev = kb - dq_slots
        if not stage_done[prev % act_slots].passes((prev // act_slots) & 1):
            return False
        if prev not in mma_done:
            raise AssertionError(f"tensor-memory slot of stage {kb} rewritten before the MMAs "
                                 f"of stage {prev} completed")
        return True

    def warp(wp) -> bool:
        kb, step = wp["kb"], wp["step"]
        if kb >= nk:
            return False
        if step == 0:
            if not code_full[kb % code_slots].passes((kb // code_slots) & 1):
                return False
            if kb not in codes_landed:
                raise AssertionError(f"codes of stage {kb} read before they landed")
            wp["step"] = 1
            return True
        if step == 1:        # slot wait before the reads (stages of four atoms)
            if slot_first and not slot_ready(kb):
                return False
            wp["step"] = 2
            return True
        if step == 2:        # codes in registers: release the code slot
            consumed.add(kb)
            code_empty[kb % code_slots].arrive(("read", kb))
            wp["step"] = 3
            return True
        if step == 3:        # slot wait after the reads (stages of one or two atoms)
            if not slot_first and not slot_ready(kb):
                return False
            wp["step"] = 4
            return True
        if step == 4:
            if not act_full[kb % act_slots].passes((kb // act_slots) & 1):
                return False
            if kb not in acts_landed:
                raise AssertionError(f"activations of stage {kb} used before they landed")
            converted.add(kb)
            dq_full[kb % dq_slots].arrive(("converted", kb))
            wp["kb"] += groups
            wp["step"] = 0
            return True
        return False

    for _ in range(max_steps):
        roles = [producer, mma_thread] + [(lambda wp=wp: warp(wp)) for wp in warps]
        rnd.shuffle(roles)
        moved = False
        for role in roles:
            if rnd.random() < 0.5:
                moved |= bool(role())
        now += 1
        events.sort(key=lambda e: (e[0], e[1]))
        while events and events[0][0] <= now:
            events.pop(0)[2]()
            moved = True
        if len(mma_done) == nk and all(w["kb"] >= nk for w in warps):
            return "ok"
        if not moved and not events:
            if not (producer() or mma_thread() or any(warp(w) for w in warps)):
                return (f"deadlock at MMA stage {mma['kb']}, producer {prod}, "
                        f"warps {[(w['g'], w['kb'], w['step']) for w in warps[::4]]}")
    return "too slow"


def simulate_persistent(ntiles: int, nk: int, code_slots: int, act_slots: int, dq_slots: int,
                        groups: int, seed: int, max_steps: int = 400_000) -> str:
    """The CTA-pair kernel's protocol (one CTA's roles; the pair's second CTA
    behaves alike): the rings run across `ntiles` tiles of `nk` stages each,
    one accumulator is handed over with accum_full (committed after a tile's
    last MMA) and accum_empty (every dequant warp arrives after storing its
    part of the tile), the MMA thread waits for accum_empty before a tile's
    first MMA, and each warp stores its part of tile i right after converting
    its first stage of a later tile (or at its end). Checks, besides the
    ring checks of `simulate`, that a tile's epilogue reads the accumulator
    only after all of the tile's MMAs and before any MMA of the next tile."""
    rnd = random.Random(seed)
    total = ntiles * nk
    code_full = [Barrier(1, f"code_full[{i}]") for i in range(code_slots)]
    code_empty = [Barrier(4, f"code_empty[{i}]") for i in range(code_slots)]
    act_full = [Barrier(1, f"act_full[{i}]") for i in range(act_slots)]
    stage_done = [Barrier(1, f"stage_done[{i}]") for i in range(act_slots)]
    dq_full = [Barrier(4, f"dq_full[{i}]") for i in range(dq_slots)]
    accum_full = Barrier(1, "accum_full")
    accum_empty = Barrier(4 * groups, "accum_empty")
    now = 0
    events: list = []
    codes_landed, acts_landed, consumed, mma_done, converted = set(), set(), set(), set(), set()
    stored = {}          # tile -> warps that stored their part
    issued_tile = [-1]   # tile of the last MMA issued

    def later(delay, fn):
        events.append((now + delay, len(events), fn))

    def land(kind, s):
        def f():
            (codes_landed if kind == "codes" else acts_landed).add(s)
            (code_full[s % code_slots] if kind == "codes" else act_full[s % act_slots]).arrive((kind, s))
        return f

    prod = {"ci": 0, "ai": 0}
    while prod["ci"] < min(total, code_slots):
        later(rnd.randint(1, 40), land("codes", prod["ci"]))
        prod["ci"] += 1

    def producer() -> bool:
        moved = False
        ci, ai = prod["ci"], prod["ai"]
        if ci < total and code_empty[ci % code_slots].passes(((ci // code_slots) & 1) ^ 1):
            if ci >= code_slots and (ci - code_slots) not in consumed:
                raise AssertionError(f"code slot of stage {ci} refilled early")
            later(rnd.randint(1, 40), land("codes", ci))
            prod["ci"] += 1
            moved = True
        if ai < total and stage_done[ai % act_slots].passes(((ai // act_slots) & 1) ^ 1):
            if ai >= act_slots and (ai - act_slots) not in mma_done:
                raise AssertionError(f"activation slot of stage {ai} refilled early")
            later(rnd.randint(1, 40), land("acts", ai))
            prod["ai"] += 1
            moved = True
        return moved

    mma = {"s": 0, "busy_until": 0}

    def mma_thread() -> bool:
        s = mma["s"]
        if s >= total:
            return False
        kb, tl = s % nk, s // nk
        if kb == 0 and tl > 0 and not accum_empty.passes((tl - 1) & 1):
            return False
        if not dq_full[s % dq_slots].passes((s // dq_slots) & 1):
            return False
        if s not in converted or s not in acts_landed:
            raise AssertionError(f"MMAs of stage {s} issued before its operands were ready")
        if kb == 0 and tl > 0 and len(stored.get(tl - 1, ())) != 4 * groups:
            raise AssertionError(f"tile {tl} overwrites the accumulator before tile {tl - 1} was stored")
        issued_tile[0] = tl
        mma["s"] += 1
        done_at = max(now, mma["busy_until"]) + rnd.randint(1, 30)
        mma["busy_until"] = done_at

        def complete(s=s, kb=kb, tl=tl):
            mma_done.add(s)
            stage_done[s % act_slots].arrive(("mma", s))
            if kb == nk - 1:
                accum_full.arrive(("tile", tl))
        events.append((done_at, len(events), complete))
        return True

    warps = [{"id": (g, i), "kb": g, "step": 0, "done": 0} for g in range(groups) for i in range(4)]

    def epilogue_step(wp, upto) -> bool:
        # store the parts of tiles [done, upto); one tile per call
        i = wp["done"]
        if i >= upto:
            return False
        if not accum_full.passes(i & 1):
            return False
        if not all(s in mma_done for s in range(i * nk, (i + 1) * nk)):
            raise AssertionError(f"tile {i} stored before its MMAs completed")
        if issued_tile[0] > i:
            raise AssertionError(f"tile {i} stored after the next tile's MMAs started")
        stored.setdefault(i, set()).add(wp["id"])
        accum_empty.arrive(("stored", i))
        wp["done"] += 1
        return True

    def warp(wp) -> bool:
        s, step = wp["kb"], wp["step"]
        if step == 9:                       # final epilogues
            return epilogue_step(wp, ntiles)
        if s >= total:
            wp["step"] = 9
            return True
        if step == 0:
            if not code_full[s % code_slots].passes((s // code_slots) & 1):
                return False
            if s not in codes_landed:
                raise AssertionError(f"codes of stage {s} read before they landed")
            consumed.add(s)
            code_empty[s % code_slots].arrive(("read", s))
            wp["step"] = 1
            return True
        if step == 1:
            if s >= dq_slots:
                prev = s - dq_slots
                if not stage_done[prev % act_slots].passes((prev // act_slots) & 1):
                    return False
                if prev not in mma_done:
                    raise AssertionError(f"tensor-memory slot of stage {s} rewritten early")
            wp["step"] = 2
            return True
        if step == 2:
            if not act_full[s % act_slots].passes((s // act_slots) & 1):
                return False
            if s not in acts_landed:
                raise AssertionError(f"activations of stage {s} used before they landed")
            converted.add(s)
            dq_full[s % dq_slots].arrive(("converted", s))
            wp["step"] = 3
            return True
        if step == 3:                       # epilogues of the tiles before s's tile
            if wp["done"] < s // nk:
                return epilogue_step(wp, s // nk)
            wp["kb"] += groups
            wp["step"] = 0
            return True
        return False

    for _ in range(max_steps):
        roles = [producer, mma_thread] + [(lambda wp=wp: warp(wp)) for wp in warps]
        rnd.shuffle(roles)
        moved = False
        for role in roles:
            if rnd.random() < 0.5:
                moved |= bool(role())
        now += 1
        events.sort(key=lambda e: (e[0], e[1]))
        while events and events[0][0] <= now:
            events.pop(0)[2]()
            moved = True
        if len(mma_done) == total and all(w["done"] == ntiles for w in warps):
            return "ok"
        if not moved and not events:
            if not (producer() or mma_thread() or any(warp(w) for w in warps)):
                return (f"deadlock at MMA stage {mma['s']}, producer {prod}, "
                        f"warps {[(w['id'], w['kb'], w['step'], w['done']) for w in warps[::4]]}")
    return "too slow"
