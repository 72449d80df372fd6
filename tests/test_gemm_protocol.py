"""Model check of the grouped FP8 GEMM's TMEM hand-off protocol (no GPU).

The kernel's MMA issuer and epilogue hand the two TMEM chunk accumulators back
and forth through mbarriers that are waited on by phase parity: a wait on
parity P passes once the barrier's completed-phase count has parity != P, so it
cannot tell phase k from phase k + 2. This test runs the protocol under random
schedules with a plain model of that rule and checks that every wait that
passes is a true one: the issuer of chunk c writes its buffer only after chunk
c - 2 has been read out, and the epilogue reads chunk c only after its MMAs are
committed. The shipped scheme (one issuer, release barriers indexed by chunk
position mod 4) must never pass a false wait; a scheme that rotates the issue
over three threads with release barriers indexed by buffer must be caught
doing so (the failure that motivated the chunk-indexed barriers).
"""
import random


class Barrier:
    """An mbarrier reduced to its completed-phase count (one arrival per phase)."""

    def __init__(self):
        self.done = 0

    def arrive(self):
        self.done += 1

    def passes(self, parity: int) -> bool:
        return (self.done & 1) != parity


def run(n_chunks: int, issuers: int, chunk_keyed: bool, rng: random.Random) -> str:
    """One random schedule: "ok", "false-pass" (some parity wait passed while its condition
    was false; the schedule may deadlock afterwards) or "deadlock" (no move left)."""
    tfull = [Barrier(), Barrier()]
    tempty = [Barrier() for _ in range(4 if chunk_keyed else 2)]
    issued = [False] * n_chunks       # MMAs issued (buffer being written)
    committed = [False] * n_chunks    # tcgen05.commit arrived
    released = [False] * n_chunks     # epilogue read the buffer out
    next_of = list(range(issuers))    # next chunk of each issuing thread (chunk c -> thread c % issuers)
    pending_commit = []
    epi = 0
    ok = True

    def release_wait(c):
        if chunk_keyed:
            if c < 2:
                return True, True
            b = tempty[(c - 2) & 3]
            return b.passes(((c - 2) >> 2) & 1), released[c - 2]
        b = tempty[c & 1]
        return b.passes(((c >> 1) & 1) ^ 1), c < 2 or released[c - 2]

    while epi < n_chunks:
        moves = []
        for t in range(issuers):
            c = next_of[t]
            if c < n_chunks and release_wait(c)[0]:
                moves.append(("issue", t))
        if pending_commit:
            moves.append(("commit", None))
        if epi < n_chunks and tfull[epi & 1].passes((epi >> 1) & 1):
            moves.append(("epilogue", None))
        if not moves:
            return "deadlock" if ok else "false-pass"
        kind, t = rng.choice(moves)
        if kind == "issue":
            c = next_of[t]
            passed, truth = release_wait(c)
            if not truth:
                ok = False                # wrote a buffer still being read
            issued[c] = True
            pending_commit.append(c)
            next_of[t] += issuers
        elif kind == "commit":
            c = pending_commit.pop(rng.randrange(len(pending_commit))) if issuers > 1 else pending_commit.pop(0)
            committed[c] = True
            tfull[c & 1].arrive()
        else:
            if not committed[epi]:
                ok = False                # read a buffer before its MMAs finished
            released[epi] = True
            (tempty[epi & 3] if chunk_keyed else tempty[epi & 1]).arrive()
            epi += 1
    return "ok" if ok else "false-pass"


def test_single_issuer_chunk_keyed_release_never_passes_a_false_wait():
    rng = random.Random(1)
    for _ in range(3000):
        assert run(24, issuers=1, chunk_keyed=True, rng=rng) == "ok"


def test_single_issuer_buffer_keyed_release_is_also_sound():
    # with one issuer in chunk order the buffer-indexed barriers were sound too
    rng = random.Random(2)
    for _ in range(3000):
        assert run(24, issuers=1, chunk_keyed=False, rng=rng) == "ok"


def test_rotated_issue_needs_chunk_keyed_release():
    rng = random.Random(3)
    assert all(run(24, issuers=3, chunk_keyed=True, rng=rng) == "ok" for _ in range(3000))
    rng = random.Random(4)
    outcomes = {run(24, issuers=3, chunk_keyed=False, rng=rng) for _ in range(300)}
    assert "false-pass" in outcomes
