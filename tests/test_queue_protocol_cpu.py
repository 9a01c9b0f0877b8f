"""The two-ended work queue shared by the 4-CTA prefill kernel and the side
kernel beside it (host model of the claim rules, checked over interleavings).

One 64-bit counter holds the pairs taken from the front of the longest-first
list (low half, by 4-CTA clusters) and the claims made from its back (high
half, by the side kernel's CTA pairs).  Each claim is one atomic add that
returns the counter's previous value (front, back):
  front claim: valid while front + min(back, side) < pairs, taking pair front;
  back claim:  valid while back < side and front + back < pairs, taking pair
               pairs - 1 - back;
where `side` is the plan's side share (the list's tail of short pairs).  A
claimer stops at its first invalid claim.  Every pair must be taken exactly
once, whatever the order of the claims, and the back claims only take pairs
of the side share."""
import random

import pytest


def _claims(n, side, front_claimers, back_claimers, rnd):
    F = B = 0
    taken = []
    alive = [("f", i) for i in range(front_claimers)] + [("b", i) for i in range(back_claimers)]
    while alive:
        who = rnd.choice(alive)
        f, b = F, B          # the atomic add's return value
        if who[0] == "f":
            F += 1
            if f + min(b, side) < n:
                taken.append(("f", f))
            else:
                alive.remove(who)
        else:
            B += 1
            if b < side and f + b < n:
                taken.append(("b", n - 1 - b))
            else:
                alive.remove(who)
    return taken


@pytest.mark.parametrize("n", [0, 1, 2, 5, 13, 40])
def test_every_pair_taken_once(n):
    rnd = random.Random(n)
    for side in sorted({0, 1, n // 2, max(n - 1, 0), n}):
        for fc, bc in ((1, 0), (1, 1), (3, 2), (36, 4), (2, 8)):
            for _ in range(200):
                taken = _claims(n, side, fc, bc, rnd)
                idx = sorted(i for _, i in taken)
                assert idx == list(range(n)), (n, side, fc, bc)
                assert all(i >= n - side for k, i in taken if k == "b"), "outside the side share"


def test_front_alone_takes_everything():
    """Without the side kernel (no back claims) the front claims take every
    pair in list order, as the 4-CTA kernel alone did."""
    taken = _claims(17, 9, 4, 0, random.Random(0))
    assert [i for _, i in taken] == list(range(17))


def test_planted_mistake_is_caught():
    """Dropping min(back, side) from the front rule lets a failed back claim
    (back past the side share) hide a pair from both ends."""
    def bad(n, side, rnd):
        F = B = 0
        taken = []
        alive = ["f", "b"]
        while alive:
            who = rnd.choice(alive)
            f, b = F, B
            if who == "f":
                F += 1
                if f + b < n:
                    taken.append(f)
                else:
                    alive.remove(who)
            else:
                B += 1
                if b < side and f + b < n:
                    taken.append(n - 1 - b)
                else:
                    alive.remove(who)
        return sorted(taken)
    rnd = random.Random(3)
    assert any(bad(10, 2, rnd) != list(range(10)) for _ in range(200))
