"""A model, on the CPU, of the stage protocol of the TMA-staged head-wise
kernels: one producer fills a ring of NST stages in item order, and two
consumer groups take alternate items (item i goes to group i % 2 and stage
i % NST, phase i // NST of that stage's full barrier).  A consumer waits for
a phase by its parity, which is only sound if the barrier cannot be two or
more phases behind the awaited one when the wait starts.  The model finds
the worst case over all interleavings the protocol allows and shows that
this holds exactly when NST is even: the reason the kernel's stage count
is even (enforced there by a static_assert)."""
import pytest


def worst_lag(nst, items=64):
    """Largest (awaited phase - completed phases) a consumer can see.

    When a group starts waiting for item j (stage s = j % nst, phase
    p = j // nst), what it knows about stage s is only what its own earlier
    items imply: the producer could not have issued item j' into stage s
    before the consumer of item j' - nst released the stage.  The last item
    this group itself took in stage s bounds how far the barrier has come;
    with no such item, nothing is known beyond phase 0 being issued."""
    worst = 0
    for j in range(items):
        g, s, p = j % 2, j % nst, j // nst
        own = [i for i in range(j) if i % 2 == g and i % nst == s]
        # the group has seen phase (own[-1] // nst) complete; the phases of
        # the other group's items in between may all still be pending
        completed = own[-1] // nst + 1 if own else 0
        worst = max(worst, p - completed)
    return worst


def parity_wait_passes(awaited, completed):
    """mbarrier.try_wait.parity: true when the current phase's parity differs
    from the awaited one, i.e. the phase of that parity has completed."""
    return (completed & 1) != (awaited & 1)


@pytest.mark.parametrize("nst", [2, 4, 6])
def test_even_stage_counts_keep_waits_within_one_phase(nst):
    assert worst_lag(nst) == 0        # the awaited phase is the next one at most


@pytest.mark.parametrize("nst", [3, 5])
def test_odd_stage_counts_let_a_group_wait_two_phases_ahead(nst):
    lag = worst_lag(nst)
    assert lag == 1                   # the barrier can be one more phase behind
    # and then the parity test mistakes the older completed phase for the
    # awaited one: the wait returns while the other group's item is loading
    awaited = 5
    assert parity_wait_passes(awaited, completed=awaited - 1)
    assert not parity_wait_passes(awaited, completed=awaited)
    assert parity_wait_passes(awaited, completed=awaited + 1)
