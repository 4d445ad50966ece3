"""Host logic of the journaled multi-branch stack (CPU): the step order, the
buffer rotation and the journal calls, driven against a fake journal that
executes copies eagerly and checks the call contract, and a fake block
that is a cheap deterministic function of its input.  The schedule must
give every branch the same result as running its blocks back to back."""
import pytest
import torch

from weight_streamed_bf16_gb300.block import BlockRunner, BlockShape


class FakeJournal:
    """Eager copies; asserts the ordering contract of include/psi.h: reload
    needs a committed entry, acquire needs a reload, and a buffer that a
    commit is still reading is written only after a fence covering it."""

    def __init__(self):
        self.entries = {}
        self.pending_reload = {}      # key -> buffer id
        self.reading = set()          # buffer ids with an unfenced commit
        self.loading = set()          # buffer ids with an unacquired reload
        self.commits = self.reloads = 0

    def commit(self, key, t):
        assert key[2] == BlockRunner.ROLE_STATE
        assert id(t) not in self.loading, "commit of a buffer whose reload is not acquired"
        self.entries[key] = t.clone()
        self.reading.add(id(t))
        self.pending_reload.pop(key, None)
        self.commits += 1

    def reload(self, key, t):
        assert key in self.entries, f"reload of {key} before its commit"
        t.copy_(self.entries[key])
        self.pending_reload[key] = id(t)
        self.loading.add(id(t))
        self.reading.discard(id(t))   # the journal orders the reload after the read
        self.reloads += 1

    def acquire(self, key):
        assert key in self.pending_reload, f"acquire of {key} without a reload"
        self.loading.discard(self.pending_reload.pop(key))

    def fence(self, t):
        self.reading.discard(id(t))

    def drop(self, key):
        del self.entries[key]


class FakeRunner(BlockRunner):
    def __init__(self, N=4, d=8):
        self.s = BlockShape(d=d, N=N)
        self.x1 = torch.empty(0)
        self.journal = None
        self.calls = []

    def forward(self, X, W, Y, flags=0, marks=None):
        j = self.journal
        assert id(X) not in j.loading, "block input read before its reload was acquired"
        assert id(Y) not in j.loading, "block output written under a pending reload"
        assert id(Y) not in j.reading, "block output written while a commit reads it"
        assert X.data_ptr() != Y.data_ptr()
        Y.copy_(X * 2 + W)            # a deterministic stand-in for block W (exact in BF16)
        self.calls.append(W)


@pytest.mark.parametrize("nblocks,nbranch", [(1, 1), (3, 1), (2, 2), (5, 3), (4, 4)])
@pytest.mark.parametrize("keep", [True, False])
@pytest.mark.parametrize("io", ["journal", "device"])
def test_branch_schedule_matches_sequential(nblocks, nbranch, keep, io):
    """io = "journal": inputs and outputs are journal entries; "device":
    branch inputs are read from, and outputs written to, device tensors."""
    run = FakeRunner()
    j = FakeJournal()
    run.journal = j
    blocks = [float(b + 1) for b in range(nblocks)]
    X = [torch.full((4, 8), float(r), dtype=torch.bfloat16) for r in range(nbranch)]
    Y = [torch.zeros_like(x) for x in X]
    if io == "journal":
        for r in range(nbranch):
            j.commit((0, r, 0), X[r])
            j.fence(X[r])
        run.run_branches(blocks, j, nbranch, keep_updated=keep)
    else:
        run.run_branches(blocks, j, nbranch, keep_updated=keep, inputs=X, outputs=Y)
    for r in range(nbranch):
        want = X[r]
        for w in blocks:
            want = want * 2 + w
        got = j.entries[(nblocks, r, 0)] if io == "journal" else Y[r]
        assert torch.equal(got, want)
    assert set(j.entries) == ({(nblocks, r, 0) for r in range(nbranch)} if io == "journal"
                              else set())
    assert len(run.calls) == nblocks * nbranch
    # resident updated state: with keep_updated one branch per block boundary
    # skips the round trip
    steps = nblocks * nbranch
    skipped = (nblocks - 1) if keep else (nblocks - 1 if nbranch == 1 else 0)
    if io == "journal":
        assert j.commits - nbranch == steps - skipped
        assert j.reloads == steps - skipped
    else:   # no commit of the outputs, no reload of the inputs
        assert j.commits == steps - skipped - nbranch
        assert j.reloads == steps - skipped - nbranch


def test_schedule_alternates_branch_order():
    run = FakeRunner()
    assert run.branch_schedule(3, 2) == [(0, 0), (0, 1), (1, 1), (1, 0), (2, 0), (2, 1)]
    assert run.branch_schedule(2, 2, keep_updated=False) == [(0, 0), (0, 1), (1, 0), (1, 1)]
