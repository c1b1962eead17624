"""CPU model of the cluster kernels' index and byte accounting, checked
before any of them runs on a GPU.

Each function restates, in plain Python, which shared-memory slots a
kernel's pushes write and how many bytes each CTA's mbarrier expects:
  cluster_tma_kernel   bulk-copy push, one-shot (multicast of the slice to
                       all N CTAs) and two-shot (partition q to CTA q);
  cluster_multi_kernel N > 16: 16-CTA clusters, CTA j acting for ranks
                       j, j + 16, ...; st.async pushes to the other CTAs,
                       plain stores for ranks of the same CTA;
  coll_multi_kernel    the four other collectives above 16 ranks;
  coll_bulk_kernel     AllGather and Broadcast up to 16 ranks by multicast
                       bulk copies.
The checks: every write lands inside the launch's stage and is made
exactly once; the bytes a CTA receives from other CTAs (or, for bulk
copies, from every copy that targets it) equal what it arms its mbarrier
with, so its wait completes exactly when the last byte lands; every slot
the epilogue reads was written; and a bulk copy never reads past the last
16-byte block that holds valid input (so never into another page).
"""
import itertools

import pytest

G = 16  # CTAs per cluster above 16 ranks


def _slices(nvec, S):
    for base in range(0, nvec, S):
        yield base, min(S, nvec - base)


def _tma(N, S, nvec, count_bytes, two):
    """cluster_tma_kernel for one message: N ranks, slice S vectors."""
    Q = S // N if two else S
    stage = N * Q
    for base, npos in _slices(nvec, S):
        writes = [dict() for _ in range(N)]
        got = [0] * N
        for r in range(N):  # the copies rank r's CTA issues
            if two:
                for q in range(N):
                    ln = min(Q, npos - q * Q) if npos > q * Q else 0
                    if ln == 0:
                        continue
                    first = (base + q * Q) * 16
                    assert first % 16 == 0 and first + ln * 16 <= nvec * 16
                    assert nvec * 16 - count_bytes < 16  # the padded tail stays in the last valid block
                    for u in range(ln):
                        slot = r * Q + u
                        assert slot < stage
                        writes[q][slot] = writes[q].get(slot, 0) + 1
                    got[q] += ln * 16
            else:
                assert (base + npos) * 16 <= nvec * 16
                for dst in range(N):  # multicast to every CTA, its own included
                    for v in range(npos):
                        slot = r * Q + v
                        assert slot < stage
                        writes[dst][slot] = writes[dst].get(slot, 0) + 1
                    got[dst] += npos * 16
        for c in range(N):
            mine = (min(Q, npos - c * Q) if npos > c * Q else 0) if two else npos
            assert got[c] == N * mine * 16  # what the CTA armed its mbarrier with
            assert all(v == 1 for v in writes[c].values())
            for q in range(N):  # the epilogue reads slot [q] positions 0..mine-1
                for u in range(mine):
                    assert writes[c].get(q * Q + u) == 1


@pytest.mark.parametrize("two", [False, True])
def test_bulk_copy_push_accounting(two):
    for N in (2, 3, 4, 5, 8, 16):
        for elem, count in itertools.product((2, 4, 8), (1, 7, 33, 257, 1000)):
            nvec = -(-count * elem // 16)
            for S in ((64 * N, 8 * N, N) if two else (1, 5, 64, 256)):
                if two and S % N:
                    continue
                _tma(N, S, nvec, count * elem, two)


def _multi(N, S, nvec, two, drop=None):
    """cluster_multi_kernel: returns nothing; asserts the accounting."""
    Q = S // G if two else S
    stage = N * Q
    for base, npos in _slices(nvec, S):
        writes = [dict() for _ in range(G)]
        got = [0] * G
        for j in range(G):
            hosted = (N - j + G - 1) // G
            for m in range(hosted):
                rank = j + m * G
                for v in range(npos):
                    if two:
                        q, u = divmod(v, Q)
                        slot = rank * Q + u
                        assert slot < stage
                        writes[q][slot] = writes[q].get(slot, 0) + 1
                        if q != j:
                            got[q] += 16
                    else:
                        for c in range(G):
                            slot = rank * Q + v
                            assert slot < stage
                            writes[c][slot] = writes[c].get(slot, 0) + 1
                            if c != j:
                                got[c] += 16
        for j in range(G):
            hosted = (N - j + G - 1) // G
            mine = (min(Q, npos - j * Q) if npos > j * Q else 0) if two else npos
            assert got[j] == (N - hosted) * mine * 16
            assert all(v == 1 for v in writes[j].values())
            for q in range(N):
                for u in range(mine):
                    assert writes[j].get(q * Q + u) == 1


def test_many_rank_allreduce_accounting():
    for N in (17, 20, 33, 40, 64):
        for nvec in (1, 3, 17, 40, 100):
            for S in (1, 5, 64):
                _multi(N, S, nvec, two=False)
            for S in (16, 32, 64):
                _multi(N, S, nvec, two=True)


def _coll_multi(op, N, S, nvec, root):
    """coll_multi_kernel for one op; asserts the accounting."""
    hosted_max = (N + G - 1) // G
    stage = {"rs": hosted_max * N * S, "ag": N * S, "rd": N * S, "bc": S}[op]
    root_cta = root % G
    for base, npos in _slices(nvec, S):
        writes = [dict() for _ in range(G)]
        got = [0] * G
        expect = [0] * G
        for j in range(G):
            hosted = (N - j + G - 1) // G
            here = j == root_cta
            expect[j] = {"rs": hosted * (N - hosted) * npos, "ag": (N - hosted) * npos,
                         "bc": 0 if here else npos, "rd": (N - hosted) * npos if here else 0}[op]
            if op == "bc":
                if here:
                    for c in range(G):
                        if c == j:
                            continue
                        for v in range(npos):
                            writes[c][v] = writes[c].get(v, 0) + 1
                            got[c] += 1
                continue
            for m in range(hosted):
                rank = j + m * G
                blocks = range(N) if op == "rs" else (0,)
                for q in blocks:
                    for u in range(npos):
                        if op == "rs":
                            c, slot = q % G, ((q // G) * N + rank) * S + u
                        elif op == "ag":
                            c, slot = None, rank * S + u
                        else:
                            c, slot = root_cta, rank * S + u
                        assert slot < stage
                        targets = range(G) if c is None else (c,)
                        for t in targets:
                            writes[t][slot] = writes[t].get(slot, 0) + 1
                            if t != j:
                                got[t] += 1
        for j in range(G):
            assert got[j] == expect[j], (op, N, S, j)
            assert all(v == 1 for v in writes[j].values())


@pytest.mark.parametrize("op", ["rs", "ag", "bc", "rd"])
def test_many_rank_collectives_accounting(op):
    for N in (17, 20, 33, 64):
        for S, nvec in ((1, 3), (5, 13), (8, 8), (7, 30)):
            for root in sorted({0, N - 1, 16 % N, N // 2}):
                _coll_multi(op, N, S, nvec, root)


def _coll_bulk(op, N, S, nvec, root):
    """coll_bulk_kernel (AllGather, Broadcast up to 16 ranks): one multicast
    copy per sender and slice, the sender's own window included."""
    stage = N * S if op == "ag" else S
    for base, npos in _slices(nvec, S):
        writes = [dict() for _ in range(N)]
        got = [0] * N
        senders = range(N) if op == "ag" else (root,)
        for r in senders:
            assert (base + npos) * 16 <= nvec * 16
            for c in range(N):
                for u in range(npos):
                    slot = (r * S if op == "ag" else 0) + u
                    assert slot < stage
                    writes[c][slot] = writes[c].get(slot, 0) + 1
                got[c] += npos * 16
        for c in range(N):
            assert got[c] == (N if op == "ag" else 1) * npos * 16  # the armed expectation
            assert all(v == 1 for v in writes[c].values())
            for q in (range(N) if op == "ag" else (0,)):
                for u in range(npos):
                    assert writes[c].get((q * S if op == "ag" else 0) + u) == 1


@pytest.mark.parametrize("op", ["ag", "bc"])
def test_bulk_copy_collectives_accounting(op):
    for N in (2, 3, 4, 8, 16):
        for S, nvec in ((1, 3), (5, 13), (64, 100), (7, 30)):
            for root in sorted({0, N - 1, N // 2}):
                _coll_bulk(op, N, S, nvec, root)
