"""A model of the tcgen05 GEMV's slot protocol (host only), checked over
random interleavings.

The kernel hands 128-K slices between warps through rings of slots, each
with a pair of mbarriers waited on by phase parity:

  activation producer  issues slice q into activation slot q % nx once the
                       slot's previous slice (q - nx) is consumed
                       (xempty); the copy lands later (xfull).
  dequant warpgroup w  takes slices q = w, w + 2, ...: waits for tensor-
                       memory slot q % ns to be free (aempty), for its
                       activation slot (xfull), reads the activations,
                       writes the A slot and arrives (afull).
  MMA warp             in slice order: waits afull, reads the A slot and the
                       activation slot, commits; the commit completes later
                       and frees both slots (aempty, xempty).

A parity wait passes when the barrier's last completed phase has the
parity asked for, so a waiter that is two phases behind passes one phase
early.  The kernel's rules that prevent it: one in-order MMA consumer, and
an activation slot count that is even (each warpgroup owns its slots) or
equal to the tensor-memory slot count 3 with the tensor-memory wait first.
The host's ring sizing (fp4gemv_plan_tc) only picks such counts.  The model
checks that those configurations never let a consumer see the wrong slice
or deadlock, and that each rule is needed: breaking it lets some
interleaving read a stale slot.
"""
import random

import pytest


class Barrier:
    """mbarrier phase bookkeeping: `done` completed phases; a wait for
    parity P passes when done's parity differs from P (initially the phase
    before phase 0, parity 1, counts as completed)."""

    def __init__(self):
        self.done = 0

    def passes(self, parity):
        return (self.done & 1) != parity


def run(nx, ns, slices, rng, x_first=False, mma_warps=1):
    """One random interleaving.  Returns 'ok', 'stale' (a consumer read a
    slot holding another slice) or 'deadlock'."""
    xfull = [Barrier() for _ in range(nx)]
    xempty = [Barrier() for _ in range(nx)]
    afull = [Barrier() for _ in range(ns)]
    aempty = [Barrier() for _ in range(ns)]
    xslot = [None] * nx   # slice whose activations the slot holds
    aslot = [None] * ns   # slice whose weights the tensor-memory slot holds

    issue_q = 0
    landing = []          # issued, not landed: (slot, slice)
    wg = [{"q": w, "step": 0} for w in range(2)]
    mma = [{"q": m} for m in range(mma_warps)]
    commits = [[] for _ in range(mma_warps)]  # per issuing thread, completing in order

    while True:
        acts = []
        if issue_q < slices:
            s = issue_q % nx
            if issue_q < nx or xempty[s].passes(((issue_q // nx) & 1) ^ 1):
                acts.append(("issue",))
        if landing:
            acts.append(("land",))
        for w, st in enumerate(wg):
            q = st["q"]
            if q >= slices:
                continue
            a, xs = q % ns, q % nx
            wait_a = aempty[a].passes(((q // ns) & 1) ^ 1)
            wait_x = xfull[xs].passes((q // nx) & 1)
            first, second = (wait_x, wait_a) if x_first else (wait_a, wait_x)
            if (st["step"] == 0 and first) or (st["step"] == 1 and second):
                acts.append(("wg", w))
        for m, st in enumerate(mma):
            q = st["q"]
            if q < slices and afull[q % ns].passes((q // ns) & 1):
                acts.append(("mma", m))
        for m in range(mma_warps):
            if commits[m]:
                acts.append(("complete", m))
        if not acts:
            done = issue_q >= slices and all(st["q"] >= slices for st in wg) and all(st["q"] >= slices for st in mma)
            return "ok" if done else "deadlock"

        act = rng.choice(acts)
        if act[0] == "issue":
            landing.append((issue_q % nx, issue_q))
            issue_q += 1
        elif act[0] == "land":
            s, q = landing.pop(rng.randrange(len(landing)))  # slots land in any order
            xslot[s] = q
            xfull[s].done += 1
        elif act[0] == "wg":
            st = wg[act[1]]
            if st["step"] == 0:
                st["step"] = 1
                continue
            q = st["q"]
            if xslot[q % nx] != q:
                return "stale"
            aslot[q % ns] = q
            afull[q % ns].done += 1
            st["q"] += 2
            st["step"] = 0
        elif act[0] == "mma":
            st = mma[act[1]]
            q = st["q"]
            if aslot[q % ns] != q or xslot[q % nx] != q:
                return "stale"
            commits[act[1]].append(q)
            st["q"] += mma_warps
        else:
            q = commits[act[1]].pop(0)
            aempty[q % ns].done += 1
            xempty[q % nx].done += 1


def outcomes(nx, ns, trials=400, slices=36, seed=0, **kw):
    rng = random.Random(seed)
    return {run(nx, ns, slices, rng, **kw) for _ in range(trials)}


# the configurations the host's ring sizing can choose
@pytest.mark.parametrize("nx,ns", [(2, 3), (3, 3), (4, 3), (2, 6), (4, 6)])
def test_allowed_slot_counts_are_sound(nx, ns):
    assert outcomes(nx, ns) == {"ok"}


def test_three_activation_slots_need_three_tensor_memory_slots():
    assert "stale" in outcomes(3, 6, trials=3000)


def test_three_activation_slots_need_the_tensor_memory_wait_first():
    assert "stale" in outcomes(3, 3, trials=3000, x_first=True)


def test_even_slot_counts_allow_either_wait_order():
    assert outcomes(4, 3, x_first=True) == {"ok"}
    assert outcomes(2, 6, x_first=True) == {"ok"}


def test_two_mma_warps_break_the_parity_waits():
    # alternate slices issued by two MMA warps: a tensor-memory slot is then
    # freed out of slice order
    assert "stale" in outcomes(4, 3, trials=3000, mma_warps=2)
