"""Models of two kernels' barrier protocols, checked under random schedules
(no GPU).  Each model restates, warp role by warp role, the waits and
arrivals of a persistent kernel in k_attn.cu -- which mbarrier each role
waits on, for which use (phase) of it, and what it arrives on -- and runs the
roles as interleaved agents with asynchronous copies and tensor-core work
completing in random order.  Checked: every wait ends only after the phase
it means has completed (never early, never a phase of the same parity two
uses later), no schedule stalls, and the work is done exactly once.

These pin the protocols' design; the kernels' own results are checked
against the oracle by the GPU tests.
"""

import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.arr, self.done = name, count, 0, 0

    def arrive(self, n=1):
        self.arr += n
        assert self.arr <= self.count, self.name
        if self.arr == self.count:
            self.arr = 0
            self.done += 1


def waitable(bar, phase):
    """try_wait.parity(phase & 1) for a waiter that means use `phase`."""
    ok = (bar.done & 1) != (phase & 1)
    if ok:
        assert bar.done > phase, ("ended early", bar.name, bar.done, phase)
    else:
        assert bar.done <= phase, ("aliased phase", bar.name, bar.done, phase)
    return ok


def run_agents(agents, pending, rnd, limit=2_000_000):
    """Interleave the agents (generators yielding while they wait) with the
    completion of pending asynchronous work (callables)."""
    alive = [True] * len(agents)
    steps = 0
    while any(alive) or pending:
        choices = [i for i in range(len(agents)) if alive[i]] + (["p"] if pending else [])
        c = rnd.choice(choices)
        if c == "p":
            pending.pop(rnd.randrange(len(pending)))()
        else:
            try:
                next(agents[c])
            except StopIteration:
                alive[c] = False
        steps += 1
        assert steps < limit, "no progress: the protocol stalls"


# ---------------------------------------------------------------------------
# attn_prefill_tc_kernel: one persistent CTA over items (query tiles) of
# n_kt key tiles each.  Producer: Q per item (after q_empty of the item
# before), K and V per key tile g into stage g & 1 (after k_empty / v_empty of
# tile g - 2).  MMA: S one key tile ahead across items (q_full before an
# item's first S, q_empty after its last), P V after p_full and v_full, the
# item's first P V after o_free of item k - 2.  Softmax: per tile s_full, the
# P buffer's pv_done of tile g - 2, sometimes the rescale's pv_done of tile
# g - 1, for a partial last tile v_full; at the item's end pv_done of its
# last tile, then o_free.
# ---------------------------------------------------------------------------
def prefill_cta(items, rnd):
    n = len(items)
    q_full, q_empty = Bar("q_full", 1), Bar("q_empty", 1)
    kf = [Bar("k_full%d" % i, 1) for i in range(2)]
    ke = [Bar("k_empty%d" % i, 1) for i in range(2)]
    vf = [Bar("v_full%d" % i, 1) for i in range(2)]
    ve = [Bar("v_empty%d" % i, 1) for i in range(2)]
    sf = [Bar("s_full%d" % i, 1) for i in range(2)]
    pf = [Bar("p_full%d" % i, 8) for i in range(2)]
    pv = [Bar("pv_done%d" % i, 1) for i in range(2)]
    of = [Bar("o_free%d" % i, 8) for i in range(2)]
    pending = []
    tensor = []  # tensor-core work in issue order: (check at completion, barriers its commits arrive on)
    # what the buffers hold, to catch a protocol that lets one overwrite data still being read
    s_read = set()   # key tiles whose S the softmax has finished reading
    p_tile = [None, None]  # the key tile whose P each P buffer holds
    pv_done_tiles = set()
    o_read = set()   # items whose output the softmax has read out of O
    first_pv = {}    # key tile -> item, for each item's first P V

    def complete_tensor():
        check, bars = tensor.pop(0)
        check()
        for bar in bars:
            bar.arrive()

    def producer():
        g = 0
        for k in range(n):
            if k >= 1:
                while not waitable(q_empty, k - 1):
                    yield
            pending.append(q_full.arrive)
            yield
            for _ in range(items[k]):
                b = g & 1
                if g >= 2:
                    while not waitable(ke[b], (g - 2) >> 1):
                        yield
                pending.append(kf[b].arrive)
                yield
                if g >= 2:
                    while not waitable(ve[b], (g - 2) >> 1):
                        yield
                pending.append(vf[b].arrive)
                yield
                g += 1

    def mma():
        st = dict(k_next=0, j_next=0, g_next=0, nkt=items[0] if n else 0)

        def issue_s(g, last):
            b = g & 1
            while not waitable(kf[b], g >> 1):
                yield

            def check():  # S buffer g & 1 last held tile g - 2, which must have been read
                assert g < 2 or g - 2 in s_read, ("S overwritten while read", g)

            tensor.append((check, [ke[b], sf[b]] + ([q_empty] if last else [])))
            pending.append(complete_tensor)
            yield

        def issue_next_s():
            if st["j_next"] == 0:
                while not waitable(q_full, st["k_next"]):
                    yield
            yield from issue_s(st["g_next"], st["j_next"] + 1 == st["nkt"])
            st["g_next"] += 1
            st["j_next"] += 1
            if st["j_next"] == st["nkt"]:
                st["j_next"] = 0
                st["k_next"] += 1
                if st["k_next"] < n:
                    st["nkt"] = items[st["k_next"]]

        if n:
            yield from issue_next_s()
        g = 0
        for k in range(n):
            for j in range(items[k]):
                if st["k_next"] < n:
                    yield from issue_next_s()
                if j == 0 and k >= 2:
                    while not waitable(of[k & 1], (k - 2) >> 1):
                        yield
                b = g & 1
                while not waitable(pf[b], g >> 1):
                    yield
                while not waitable(vf[b], g >> 1):
                    yield
                if j == 0:
                    first_pv[g] = k

                def check(g=g):
                    assert p_tile[g & 1] == g, ("P V read another tile's P", g, p_tile)
                    if g in first_pv and first_pv[g] >= 2:  # the item's first P V overwrites O
                        assert first_pv[g] - 2 in o_read, ("O overwritten before it was read", first_pv[g])
                    pv_done_tiles.add(g)

                tensor.append((check, [ve[b], pv[b]]))
                pending.append(complete_tensor)
                yield
                g += 1

    def softmax():
        # an item's output is read out after the next item's first P is written
        # (O has two buffers), so that P V's of the next item run meanwhile
        def epilogue(k, g_last):
            while not waitable(pv[g_last & 1], g_last >> 1):
                yield
            assert g_last in pv_done_tiles, ("O read before the item's last P V", k)
            o_read.add(k)
            of[k & 1].arrive(8)
            yield

        g = 0
        late = None  # (item, its last key tile) whose output is still to be read
        for k in range(n):
            for j in range(items[k]):
                b = g & 1
                while not waitable(sf[b], g >> 1):
                    yield
                if g >= 2:
                    while not waitable(pv[b], (g - 2) >> 1):
                        yield
                if j >= 1 and rnd.random() < 0.3:  # a row's max grew: O is rescaled
                    while not waitable(pv[(g - 1) & 1], (g - 1) >> 1):
                        yield
                if j == items[k] - 1 and rnd.random() < 0.5:  # a partial last tile: zero V rows
                    while not waitable(vf[b], g >> 1):
                        yield
                s_read.add(g)
                assert g < 2 or g - 2 in pv_done_tiles, ("P overwritten while read", g)
                p_tile[b] = g
                pf[b].arrive(8)
                yield
                g += 1
                if j == 0 and late is not None:
                    yield from epilogue(*late)
                    late = None
            late = (k, g - 1)
        if late is not None:
            yield from epilogue(*late)

    return [producer(), mma(), softmax()], pending


@pytest.mark.parametrize("seed", range(6))
def test_prefill_persistent_protocol(seed):
    rnd = random.Random(seed)
    for _ in range(60):
        items = [rnd.randint(1, 6) for _ in range(rnd.randint(0, 7))]
        agents, pending = prefill_cta(items, rnd)
        run_agents(agents, pending, rnd)


# ---------------------------------------------------------------------------
# attn_decode_mma_kernel with work claimed at run time: G CTAs share the
# counters [next item, CTAs done].  A CTA's first item is dealt (entry
# blockIdx.x); its producer claims the rest after the grid wait, two items
# ahead, hands item j's id to the consumers through entry (j - 1) % 8 of an
# id ring (one mbarrier per entry) before the item before it starts, and
# streams every item's stages through a 3-slot ring.  The four consumer warps
# read the next id at an item's start, drain its stages and pass the item to
# the two merge warps through a 4-entry queue; two entries with no item end
# the merge warps.  The last CTA to finish claiming resets the counters.
# ---------------------------------------------------------------------------
def decode_grid(total, G, stages_of, dynamic, rnd, claim, consumed, merged):
    S, K_IDS, K_MERGE, NC, NM = 3, 8, 4, 4, 2
    agents, pending = [], []
    for b in range(G):
        full = [Bar("full%d" % i, 1) for i in range(S)]
        empty = [Bar("empty%d" % i, NC) for i in range(S)]
        idf = [Bar("id%d" % i, 1) for i in range(K_IDS)]
        ids = [None] * K_IDS
        mfull = [Bar("mfull%d" % i, NC) for i in range(K_MERGE)]
        mempty = [Bar("mempty%d" % i, 1) for i in range(K_MERGE)]
        mq = [None] * K_MERGE
        slot = [None] * S

        def cta(b=b, full=full, empty=empty, idf=idf, ids=ids, mfull=mfull, mempty=mempty, mq=mq, slot=slot):
            def nth(k):
                return k * G + ((G - 1 - b) if (k & 1) else b)

            def producer():
                def take(j):
                    if not dynamic:
                        return nth(j)
                    v = G + claim[0]
                    claim[0] += 1
                    if v >= total:
                        claim[1] += 1
                        if claim[1] == G:
                            claim[0] = claim[1] = 0
                    return v

                def publish(j, v):
                    ids[(j - 1) % K_IDS] = v
                    idf[(j - 1) % K_IDS].arrive()

                g = issued = 0
                waited = False
                nxt = nxt2 = total
                q, k = b, 0
                while q < total:
                    if k >= 1:
                        nxt = nxt2
                        publish(k + 1, nxt)
                        yield
                        nxt2 = take(k + 2) if nxt < total else total
                        yield
                    for t in range(stages_of(q)):
                        if not waited and (issued >= S or rnd.random() < 0.3):
                            waited = True
                            nxt = take(1)
                            publish(1, nxt)
                            yield
                            nxt2 = take(2) if nxt < total else total
                            yield
                        s = g % S
                        while (empty[s].done & 1) == (((g // S) & 1) ^ 1):  # the release of use g // S - 1
                            yield
                        slot[s] = (q, t)
                        pending.append(full[s].arrive)
                        yield
                        issued += 1
                        g += 1
                    if not waited:
                        waited = True
                        nxt = take(1)
                        publish(1, nxt)
                        yield
                        nxt2 = take(2) if nxt < total else total
                        yield
                    q, k = nxt, k + 1

            def consumer(w):
                g = k = 0
                q = b
                while q < total:
                    while not waitable(idf[k % K_IDS], k // K_IDS):
                        yield
                    q_nx = ids[k % K_IDS]
                    for t in range(stages_of(q)):
                        s = g % S
                        while not waitable(full[s], g // S):
                            yield
                        assert slot[s] == (q, t)
                        if w == 0:
                            consumed.append((q, t))
                        empty[s].arrive()
                        yield
                        g += 1
                    e = k % K_MERGE
                    if k >= K_MERGE:
                        while not waitable(mempty[e], k // K_MERGE - 1):
                            yield
                    if w == 0:
                        mq[e] = q
                    mfull[e].arrive()
                    yield
                    q, k = q_nx, k + 1
                for kk in range(k, k + NM):
                    e = kk % K_MERGE
                    if kk >= K_MERGE:
                        while not waitable(mempty[e], kk // K_MERGE - 1):
                            yield
                    if w == 0:
                        mq[e] = -1
                    mfull[e].arrive()
                    yield

            def merger(mw):
                k = mw
                while True:
                    e = k % K_MERGE
                    while not waitable(mfull[e], k // K_MERGE):
                        yield
                    if mq[e] < 0:
                        return
                    merged.append(mq[e])
                    mempty[e].arrive()
                    yield
                    k += NM

            return [producer()] + [consumer(w) for w in range(NC)] + [merger(m) for m in range(NM)]

        agents += cta()
    return agents, pending


@pytest.mark.parametrize("dynamic", [True, False])
@pytest.mark.parametrize("seed", range(4))
def test_decode_claim_protocol(seed, dynamic):
    rnd = random.Random(1000 * seed + dynamic)
    for _ in range(12):
        G = rnd.randint(1, 6)
        total = rnd.randint(G, 14 * G)  # up to a dozen items and more per CTA: the id ring wraps
        st = [rnd.randint(1, 5) for _ in range(total)]
        claim, consumed, merged = [0, 0], [], []
        agents, pending = decode_grid(total, G, lambda q: st[q], dynamic, rnd, claim, consumed, merged)
        run_agents(agents, pending, rnd)
        assert sorted(consumed) == sorted((q, t) for q in range(total) for t in range(st[q]))
        assert sorted(merged) == list(range(total))
        assert claim == [0, 0]  # reset by the last CTA to finish claiming
