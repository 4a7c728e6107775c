"""A model of the prep pass's hand-over protocol between its two warp groups.

The prep kernel (csrc/gdn_prefill_split.cu, prep_kernel) splits into two groups
of four warps after the q/k conv.  Step g of group e is value head g when
g % 2 == e, else the v conv of value head g.  Two resources pass between the
groups:

  - staging block 1: the q rows (load 0), then the v rows of value heads 0, 1,
    ... in turn (load g + 1), each load issued by whoever read the previous
    one; a reader waits for a shared issue counter, then on the block's
    mbarrier with parity (g + 1) & 1;
  - the W^T TMEM columns: value head g's product is issued once a shared count
    of heads whose W^T has been read out reaches g.

An mbarrier parity wait is only unambiguous while the barrier is at most one
phase past the awaited completion.  This model runs the two groups and the
asynchronous landing of loads under random interleavings and checks that
every wait that succeeds sees exactly the completion it is after, that the
resources are used in head order, and that every schedule finishes.  It is a
check of the protocol's design on the host, not of the kernel.
"""
import random

import pytest


class Block:
    """Staging block 1 and its mbarrier: loads land in issue order."""

    def __init__(self):
        self.issued = 1            # the q rows, issued at kernel start
        self.landed = 0            # completed phases of the mbarrier
        self.contents = ["q"]      # what each load carries, by load index

    def issue(self, what):
        assert self.landed == self.issued, "a load was issued over one still in flight"
        self.contents.append(what)
        self.issued += 1

    def parity_done(self, k):
        """try_wait.parity on completion k: true when the current phase's parity
        differs from k's (the hardware test), checked against the true state."""
        hw = (self.landed & 1) != (k & 1)
        assert self.landed in (k, k + 1), f"parity wait for completion {k} at phase {self.landed}"
        return hw


def run(G, seed):
    rnd = random.Random(seed)
    blk = Block()
    w_read = 0                     # heads whose W^T was read out of TMEM
    w_busy = None                  # head whose product holds the W^T columns
    read_by = {}                   # load index -> group that read it
    events = []

    def group(e):
        nonlocal w_read, w_busy
        # the q rows: every thread waits, then a barrier of the whole CTA
        while not blk.parity_done(0):
            yield
        yield "barrier"
        for _ in range(rnd.randint(1, 3)):
            yield                  # the q conv
        if e == 0:
            blk.issue("v0")        # the last warp done with the q rows (release_q)
        yield "barrier"            # the k conv, the Gram product and the K^ tile, then the split
        for g in range(G):
            if g % 2 != e:
                # v conv of head g: its rows are load g + 1, issued as the (g + 2)-th load
                while blk.issued < g + 2:
                    yield
                while not blk.parity_done(g + 1):
                    yield
                assert blk.contents[g + 1] == f"v{g}"
                read_by[g + 1] = e
                for _ in range(rnd.randint(1, 4)):
                    yield          # the conv itself
                events.append(("vconv", g, e))
                if g + 1 < G:
                    blk.issue(f"v{g + 1}")
            else:
                for _ in range(rnd.randint(1, 6)):
                    yield          # A, P, the solve, T diag(beta)
                while w_read < g:
                    yield
                assert w_busy is None, "two W^T products in the same columns"
                w_busy = g
                for _ in range(rnd.randint(1, 3)):
                    yield          # the product
                assert w_busy == g
                w_busy = None
                w_read += 1
                events.append(("head", g, e))

    gens = [group(0), group(1)]
    arrived = [0, 0]               # CTA barriers each group has reached
    waiting = [False, False]       # the group's last step was arriving at a barrier
    done = [False, False]
    steps = 0
    while not all(done):
        steps += 1
        assert steps < 100000, "no progress: deadlock"
        choices = [i for i in range(2) if not done[i]]
        if blk.landed < blk.issued:
            choices.append("land")
        c = rnd.choice(choices)
        if c == "land":
            blk.landed += 1
            continue
        # a CTA barrier: neither group passes it before the other has reached it
        if waiting[c] and arrived[1 - c] < arrived[c]:
            continue
        waiting[c] = False
        try:
            if next(gens[c]) == "barrier":
                arrived[c] += 1
                waiting[c] = True
        except StopIteration:
            done[c] = True
    return events, read_by, w_read, blk


@pytest.mark.parametrize("G", [1, 2, 3, 4])
def test_prep_group_protocol(G):
    for seed in range(300):
        events, read_by, w_read, blk = run(G, seed)
        heads = [g for kind, g, _ in events if kind == "head"]
        vconvs = [g for kind, g, _ in events if kind == "vconv"]
        assert heads == list(range(G)), "W^T products out of head order"
        assert sorted(vconvs) == list(range(G))
        assert vconvs == sorted(vconvs), "v rows read out of head order"
        assert w_read == G
        assert blk.issued == G + 1 and blk.landed == G + 1
        for g in range(G):   # head g's v conv on the other group than head g itself
            assert read_by[g + 1] == 1 - (g % 2)
