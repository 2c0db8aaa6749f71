"""Model check of the key ring's barrier protocol (host-side model, no GPU).

The L1-norm kernel moves each 128-key tile through a ring of S shared-memory
stages (8 stages per tile, stage n in slot n % S).  Producer groups fill the
stages: with g groups, group i fills the stages n with n % g == i, one stage
at a time, each stage's copies landing after a variable delay (a lane's
cp.async.mbarrier.arrive.noinc holds the group until they have).  Two MMA
issuers consume them: issuer H takes the stages n with n % 2 == H, in order,
and tests the next stage's barrier before issuing the current stage's MMAs.
A stage's slot is freed (empty barrier) when the issuer's MMAs on it have
completed; the tensor pipe runs MMAs one at a time in issue order.

mbarrier waits and tests are by phase parity: a wait for parity P succeeds
when the barrier's number of completed phases c has (c & 1) != P.  It is
unambiguous only if the barrier is at most one phase away from the phase the
thread wants; a barrier two phases behind passes the test too early.  The
kernel keeps the ring depth even (and at least the number of groups), which
makes that impossible: the stage one ring-length before the one an issuer
tests has the issuer's own parity, so the issuer has already acquired it.
This model runs the protocol under random delays and checks every successful
wait or test against the phase it was meant to see: never wrong with an even
depth (or with one group), and wrong for some schedules with an odd depth
and two groups.
"""

import heapq
import random

import pytest


def simulate(S, groups, tiles, seed, stall_prob=0.08, issuers=2, wide=False):
    """Run the ring protocol once; return (violations, stages consumed).
    Issuer h takes the stages n with n % issuers == h.  With ``wide`` every
    group fills its part of every stage, in order (the CTA-pair kernel's
    32 KB stages): a slot's full phase completes when all groups landed."""
    rng = random.Random(seed)
    N = 8 * tiles
    full = [0] * S    # completed phases of each slot's full barrier
    empty = [0] * S   # completed phases of each slot's empty barrier
    violations = []
    events = []       # (time, seq, kind, payload)
    seq = [0]

    def push(t, kind, payload):
        seq[0] += 1
        heapq.heappush(events, (t, seq[0], kind, payload))

    def delay(base):
        d = base * (0.5 + rng.random())
        if rng.random() < stall_prob:
            d *= 4 + 12 * rng.random()   # a slow L2 round trip or a descheduled warp
        return d

    def passes(count, parity):
        return (count & 1) != parity

    prod_next = {g: (0 if wide else g) for g in range(groups)}  # next stage of each producer group
    arrivals = [[] for _ in range(S)]  # wide: stages of the groups that landed in the open phase
    iss_next = {h: h for h in range(issuers)}      # next stage of each issuer
    iss_ready = {h: False for h in range(issuers)}  # next stage already acquired by a test
    pipe_free = [0.0]
    consumed = [0]
    for g in range(groups):
        push(0.0, "prod", g)
    for h in range(issuers):
        push(0.0, "iss", h)

    steps = 0
    while events and steps < 200000:
        steps += 1
        t, _, kind, who = heapq.heappop(events)
        if kind == "prod":
            n = prod_next[who]
            if n >= N:
                continue
            s, u = n % S, n // S
            # wait for the slot's empty barrier: phase u - 1 (its previous use) completed
            if passes(empty[s], (u & 1) ^ 1):
                if empty[s] != u:
                    violations.append(("producer", n, empty[s], u))
                push(t + delay(600.0), "landed", (who, n))
            else:
                push(t + 20.0, "prod", who)
        elif kind == "landed":
            g, n = who
            if wide:
                a = arrivals[n % S]
                if a and a[0] != n:
                    violations.append(("mixed phase", n, a[0], n))
                a.append(n)
                if len(a) == groups:
                    full[n % S] += 1
                    a.clear()
                prod_next[g] = n + 1
            else:
                full[n % S] += 1
                prod_next[g] = n + groups
            push(t + 5.0, "prod", g)   # the group moves on once its copies have landed
        elif kind == "iss":
            n = iss_next[who]
            if n >= N:
                continue
            s, u = n % S, n // S
            if not iss_ready[who]:
                if not passes(full[s], u & 1):
                    push(t + 20.0, "iss", who)
                    continue
                if full[s] != u + 1:
                    violations.append(("issuer wait", n, full[s], u + 1))
            # test the next own stage before issuing this one's MMAs
            m = n + issuers
            iss_ready[who] = False
            if m < N:
                sm, um = m % S, m // S
                if passes(full[sm], um & 1):
                    iss_ready[who] = True
                    if full[sm] != um + 1:
                        violations.append(("issuer test", m, full[sm], um + 1))
            start = max(t + 40.0, pipe_free[0])
            pipe_free[0] = start + 256.0 * (0.9 + 0.2 * rng.random())
            push(pipe_free[0], "mma_done", n)
            iss_next[who] = n + issuers
            push(t + delay(400.0 * issuers / 2), "iss", who)
        elif kind == "mma_done":
            empty[who % S] += 1
            consumed[0] += 1
    return violations, consumed[0]


@pytest.mark.parametrize("stall_prob", [0.08, 0.3])
@pytest.mark.parametrize("S", [4, 6, 8, 10, 12])
@pytest.mark.parametrize("groups", [1, 2, 4])
def test_even_ring_depth_never_tests_a_barrier_two_phases_behind(S, groups, stall_prob):
    if groups > S:
        pytest.skip("the ring holds at least as many stages as there are groups")
    for seed in range(20):
        violations, consumed = simulate(S, groups, tiles=30, seed=1000 * S + 10 * groups + seed,
                                        stall_prob=stall_prob)
        assert violations == [], (S, groups, seed, violations[:3])
        assert consumed == 8 * 30, "every stage is consumed (no deadlock)"


@pytest.mark.parametrize("S", [5, 7, 9, 11])
def test_odd_ring_depth_with_one_group_is_safe(S):
    for seed in range(20):
        violations, consumed = simulate(S, 1, tiles=30, seed=7000 + 10 * S + seed, stall_prob=0.3)
        assert violations == [] and consumed == 240


@pytest.mark.parametrize("S", [5, 7, 9])
def test_odd_ring_depth_with_two_groups_can_pass_a_test_early(S):
    """Why the host never picks an odd depth: with two producer groups, one
    of them slowed down, an issuer can find a slot's full barrier (or a
    producer its empty barrier) two phases behind, i.e. take a stage that has
    not been filled (or overwrite one still being read)."""
    found = []
    for seed in range(40):
        violations, _ = simulate(S, 2, tiles=30, seed=9000 + 10 * S + seed, stall_prob=0.3)
        found += violations
        if found:
            break
    assert found, "expected an early pass with an odd ring depth and two groups"
    kind, n, seen, wanted = found[0]
    assert seen == wanted - 2, "the barrier was two phases behind"


@pytest.mark.parametrize("S", [4, 6, 8, 10, 12])
@pytest.mark.parametrize("groups", [1, 2])
def test_four_issuers_with_one_or_two_groups_and_an_even_depth_are_safe(S, groups):
    """Four MMA issuers (each owning every fourth stage, as the L1-norm launch
    runs them when the heads fit in 64 accumulator columns).  An issuer about
    to take stage m holds stage m - 4; the slot's previous stage m - S has the
    parity of m - 4 whenever S is even, so with one or two producer groups
    (each filling its stages in order) it was filled before m - 4: no barrier
    is ever two phases behind.  The general rule: S = issuers (mod groups)."""
    for seed in range(20):
        violations, consumed = simulate(S, groups, tiles=30, seed=11000 + 10 * S + groups + seed,
                                        stall_prob=0.3, issuers=4)
        assert violations == [], (S, groups, seed, violations[:3])
        assert consumed == 240


def test_four_issuers_and_four_groups_need_a_depth_multiple_of_four():
    """With four producer groups as well, six slots break the rule: stage
    m - 6 belongs to another group and can still be unfilled."""
    found = []
    for seed in range(80):
        violations, _ = simulate(6, 4, tiles=30, seed=12000 + seed, stall_prob=0.3, issuers=4)
        found += violations
        if found:
            break
    assert found, "expected an early pass with four groups, four issuers and six slots"
    kind, n, seen, wanted = found[0]
    assert seen == wanted - 2
    for seed in range(20):
        violations, consumed = simulate(8, 4, tiles=30, seed=12500 + seed, stall_prob=0.3, issuers=4)
        assert violations == [] and consumed == 240


@pytest.mark.parametrize("S", [2, 3, 4, 5, 6, 7])
def test_wide_stages_filled_by_every_group_in_order_are_safe_at_any_depth(S):
    """The CTA-pair kernel's ring: each 32 KB stage is filled by both producer
    groups (one half each), every group in stage order, and two issuers take
    alternate stages.  A stage is full only once every group landed it, and
    each group lands its stages in order, so when an issuer's previous stage
    is full so is every earlier one: no barrier is two phases behind, odd
    depths included (the kernel runs five)."""
    for seed in range(20):
        violations, consumed = simulate(S, 2, tiles=30, seed=13000 + 10 * S + seed, stall_prob=0.3, wide=True)
        assert violations == [], (S, seed, violations[:3])
        assert consumed == 240
