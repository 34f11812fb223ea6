"""A model of the grouped GEMM's hand-offs (csrc/q4_moe_gemm.cu) for the rule
under which its MMA issuers may take their K steps in pairs behind one wait.

Roles, each in K-step order: the TMA thread fills input stage k % IS once
stage k - IS is empty; the dispatch thread releases step k once its input
landed and A stage k % AS is free (the MMAs of step k - AS done); the dequant
warps write A stage k % AS and release the input stage; an issuer issues its
steps (all of them in GLU mode, every other one in plain mode), the MMA of a
step emptying its input and A stages.  With pairing an issuer holds its first
step until its next one is dequantised.  The kernel pairs only with 4 A
stages and, in plain mode, 3 or more input stages; the model finds no
deadlock under that rule and one outside it (plain mode with 2 input stages,
or 2 A stages)."""
import itertools

import pytest


def run(IS, AS, n, glu, pairing):
    in_full, deq_done, mma_done, a_full, go = set(), set(), set(), set(), set()
    tma = disp = deq = 0
    own = [[k for k in range(n) if glu or (k & 1) == r] for r in (0, 1)]
    pos, pend = [0, 0], [None, None]
    progress = True
    while progress:
        progress = False
        if tma < n and (tma < IS or (tma - IS in deq_done and tma - IS in mma_done)):
            in_full.add(tma)
            tma += 1
            progress = True
        if disp < n and disp in in_full and (disp < AS or disp - AS in mma_done):
            go.add(disp)
            disp += 1
            progress = True
        if deq < n and deq in go:
            deq_done.add(deq)
            a_full.add(deq)
            deq += 1
            progress = True
        for r in (0, 1):
            if pos[r] >= len(own[r]):
                continue
            k = own[r][pos[r]]
            if pairing and pend[r] is None and pos[r] + 1 < len(own[r]):
                pend[r] = k
                pos[r] += 1
                progress = True
                continue
            if k in a_full:
                if pend[r] is not None:
                    mma_done.add(pend[r])
                    pend[r] = None
                mma_done.add(k)
                pos[r] += 1
                progress = True
    return len(mma_done) == n and deq == n


def kernel_rule(IS, AS, glu):
    return AS >= 4 and (glu or IS >= 3)


@pytest.mark.parametrize("glu", [False, True])
def test_pairing_rule_never_deadlocks(glu):
    for n, IS, AS in itertools.product(range(1, 48), range(2, 17), (2, 3, 4)):
        assert run(IS, AS, n, glu, kernel_rule(IS, AS, glu)), (n, IS, AS, glu)


def test_without_pairing_never_deadlocks():
    for n, IS, AS, glu in itertools.product(range(1, 48), range(2, 17), (2, 3, 4), (False, True)):
        assert run(IS, AS, n, glu, False), (n, IS, AS, glu)


def test_the_excluded_cases_do_deadlock():
    assert not run(2, 4, 101, False, True)  # plain mode, 2 input stages
    assert not run(3, 2, 101, False, True)  # 2 A stages
    assert run(2, 4, 101, True, True)       # GLU mode pairs with 2 input stages
