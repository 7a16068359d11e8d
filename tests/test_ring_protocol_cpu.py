"""A model of the staged row kernel's copy ring, checked for every stage count
and row count (no GPU).

The kernel (csrc/kernels.cuh, staged_kernel) streams a CTA's rows through S
shared-memory stages.  Row r always goes to stage r mod S (thread 0 issues
copies in row order and advances the stage by counting).  Thread 0 issues the
first S-1 rows before the loop and one more row right after the first
barrier of each iteration; at that barrier every thread has finished the
previous iteration, so the rows it was done with are free.

What a wait on a row that was never issued would mean on the GPU is a bounded
wait running out (the kernel then flags an error and returns): the model
checks that this never happens, and that no copy is issued into a stage whose
row some thread may still read.
"""
import pytest


def run_ring(S, nrows, pipelined_stats):
    """Replay one CTA's loop.  pipelined_stats: the LayerNorm forward, which
    during iteration k reads row k (variance, output) and row k+1 (sum), and
    waits for row k+1 in iteration k.  Returns the issue order."""
    issued = []

    def issue():
        r = len(issued)
        if r < nrows:
            issued.append(r)

    def wait(r):
        assert r < len(issued), f"S={S} nrows={nrows}: wait for row {r} before its copy was issued"

    while len(issued) < min(nrows, S - 1):
        issue()
    for k in range(nrows):
        if not pipelined_stats or k == 0:
            wait(k)
        if pipelined_stats and k + 1 < nrows:
            wait(k + 1)            # before this iteration's barrier
        # first barrier of iteration k: every thread is done with the rows
        # below `oldest_live`; the next copy goes to stage issued mod S
        oldest_live = k            # rows >= k may still be read (row k after the barrier)
        r = len(issued)
        if r < nrows:
            assert r - S < oldest_live, (
                f"S={S} nrows={nrows}: row {r} would overwrite stage of row {r - S} still in use")
        issue()
    assert issued == list(range(nrows))
    return issued


@pytest.mark.parametrize("S", range(2, 17))
def test_ring_one_row_per_iteration(S):
    for nrows in range(1, 3 * S + 5):
        run_ring(S, nrows, pipelined_stats=False)


@pytest.mark.parametrize("S", range(3, 17))
def test_ring_layernorm_forward_pipelined(S):
    for nrows in range(1, 3 * S + 5):
        run_ring(S, nrows, pipelined_stats=True)


def test_layernorm_forward_needs_three_stages():
    # with two stages, the wait for row 1 in iteration 0 comes before the
    # copy of row 1 is issued (it is issued at that iteration's barrier): the
    # launcher gives the LayerNorm forward at least three stages
    with pytest.raises(AssertionError, match="before its copy was issued"):
        run_ring(2, 4, pipelined_stats=True)
    run_ring(3, 4, pipelined_stats=True)
