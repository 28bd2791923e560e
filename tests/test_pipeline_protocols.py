"""The kernels' mbarrier protocols, checked on the host under many random schedules
(race detection without compute-sanitizer).  Each model mirrors a kernel's roles line
for line as far as synchronisation goes: what each role waits on, in which order, which
barrier (and which completion of it) each wait targets, what it arrives on or commits
to, and which buffer each copy or MMA reads or writes.  Under every schedule the model
checks: no deadlock; no parity wait that could see the wrong phase; no arrival beyond a
barrier's count; and every buffer holding what its reader expects (no overwrite before
the last read, no read before the write).  Mutation tests plant the protocol mistakes
these checks are for and require that the model catches each of them.

Models: the prefill attention CTA (Q/K loader, V loader, Q K^T issuer, P V issuer, four
softmax warps; two-deep K, V and S/P rings with per-parity barriers; the sink strip as
tile 0; the lazy O rescale), and the decode split block (one producer lane, consumer
warps over a STAGES-deep ring, the end-of-block drain; and for the decode step, the
token warp, its ring of two rotated q rows and the barrier that holds back the tile
holding the token's new row)."""
import random
import re

import pytest

from tests.pipeline_model import Barrier, Deadlock, ProtocolError, run

# --------------------------------------------------------------------------- prefill


def prefill_roles(n, n_strip, rescale, mutate=None):
    """One prefill CTA visiting n key tiles (tile 0 a sink strip when n_strip).
    rescale[(w, i)]: softmax warp w rescales O at tile i (a row max grew)."""
    B = Barrier
    q_full = B("q_full", 1)
    k_full = [B(f"k_full{s}", 1) for s in range(2)]
    k_empty = [B(f"k_empty{s}", 1) for s in range(2)]
    v_full = [B(f"v_full{s}", 1) for s in range(2)]
    v_empty = [B(f"v_empty{s}", 1) for s in range(2)]
    s_full = [B(f"s_full{s}", 1) for s in range(2)]
    if mutate == "one_p_barrier":
        shared = B("p_full", 4)
        p_full = [shared, shared]
    else:
        p_full = [B(f"p_full{s}", 4) for s in range(2)]
    pv_done = [B(f"pv_done{s}", 1) for s in range(2)]
    if mutate == "one_p_barrier":
        p_index = lambda i: i          # a single barrier completes once per tile
    else:
        p_index = lambda i: i >> 1     # per-parity barriers complete every second tile

    st = {"q": None, "k": [None, None], "v": [None, None], "s": [[None] * 4 for _ in range(2)],
          "o": [None] * 4, "qk_done": set(), "pv_done": set()}

    def fail(msg):
        raise ProtocolError(msg)

    def loader_qk():
        yield ("expect", q_full, 1)
        yield ("tma", q_full, 1, lambda: st.__setitem__("q", "Q"))
        for i in range(n):
            s = i & 1
            if i >= 2 and mutate != "no_k_empty_wait":
                yield ("wait", k_empty[s], (i >> 1) - 1)

            def issue(i=i):
                if i >= 2 and i - 2 not in st["qk_done"]:
                    fail(f"K{i} copied over K{i - 2} before Q K^T{i - 2} ran")
            yield ("do", issue)
            yield ("expect", k_full[s], 1)
            yield ("tma", k_full[s], 1, lambda s=s, i=i: st["k"].__setitem__(s, ("K", i)))

    def loader_v():
        for i in range(n):
            s = i & 1
            if i >= 2:
                yield ("wait", v_empty[s], (i >> 1) - 1)

            def issue(i=i):
                if i >= 2 and i - 2 not in st["pv_done"]:
                    fail(f"V{i} copied over V{i - 2} before P V{i - 2} ran")
            yield ("do", issue)
            yield ("expect", v_full[s], 1)
            yield ("tma", v_full[s], 1, lambda s=s, i=i: st["v"].__setitem__(s, ("V", i)))

    def qk_issuer():
        yield ("wait", q_full, 0)
        for i in range(n):
            s = i & 1
            yield ("wait", k_full[s], i >> 1)
            if i >= 2 and mutate != "no_pv_wait_before_qk":
                yield ("wait", pv_done[s], (i >> 1) - 1)

            def mma(i=i, s=s):
                if st["q"] != "Q" or st["k"][s] != ("K", i):
                    fail(f"Q K^T{i} read {st['q']}, {st['k'][s]}")
                if i >= 2 and i - 2 not in st["pv_done"]:
                    fail(f"Q K^T{i} overwrote P{i - 2} before P V{i - 2} read it")
                for w in range(4):
                    st["s"][s][w] = ("S", i)
                st["qk_done"].add(i)
            yield ("mma", "qk", mma)
            yield ("commit", "qk", s_full[s])
            yield ("commit", "qk", k_empty[s])

    def pv_issuer():
        for j in range(n):
            s = j & 1
            yield ("wait", p_full[s], p_index(j))
            yield ("wait", v_full[s], j >> 1)
            steps = 1 if j < n_strip else 4   # the strip is one K step; a full tile four
            for kk in range(steps):
                def mma(j=j, s=s, kk=kk, last=kk == steps - 1):
                    for w in range(4):
                        if st["s"][s][w] != ("P", j):
                            fail(f"P V{j} read {st['s'][s][w]} in rows of warp {w}")
                        want = ("O", j - 1) if kk == 0 else ("Opart", j, kk - 1)
                        if (j > 0 or kk > 0) and st["o"][w] != want:
                            fail(f"P V{j} step {kk} accumulated onto {st['o'][w]}")
                    if st["v"][s] != ("V", j):
                        fail(f"P V{j} read {st['v'][s]}")
                    for w in range(4):
                        st["o"][w] = ("O", j) if last else ("Opart", j, kk)
                    if last:
                        st["pv_done"].add(j)
                yield ("mma", "pv", mma)
            yield ("commit", "pv", pv_done[s])
            yield ("commit", "pv", v_empty[s])

    def softmax(w):
        for i in range(n):
            s = i & 1
            yield ("wait", s_full[s], i >> 1)

            def read_s(i=i, s=s):
                if st["s"][s][w] != ("S", i):
                    fail(f"softmax {w} read {st['s'][s][w]} for S{i}")
            yield ("do", read_s)
            if i >= n_strip and i > 0 and rescale[(w, i)]:
                # O is rescaled after P V of the previous tile is done
                yield ("wait", pv_done[(i - 1) & 1], (i - 1) >> 1)

                def rescale_o(i=i):
                    if st["o"][w] != ("O", i - 1):
                        fail(f"softmax {w} rescaled O holding {st['o'][w]} at tile {i}")
                yield ("do", rescale_o)
            yield ("do", lambda i=i, s=s: st["s"][s].__setitem__(w, ("P", i)))
            yield ("arrive", p_full[s])
        yield ("wait", pv_done[(n - 1) & 1], (n - 1) >> 1)

        def epilogue():
            if st["o"][w] != ("O", n - 1):
                fail(f"epilogue {w} read {st['o'][w]}")
        yield ("do", epilogue)

    roles = {"loader_qk": loader_qk(), "loader_v": loader_v(), "qk": qk_issuer(), "pv": pv_issuer()}
    for w in range(4):
        roles[f"softmax{w}"] = softmax(w)
    return roles


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 9])
@pytest.mark.parametrize("n_strip", [0, 1])
@pytest.mark.parametrize("p_rescale", [0.0, 0.3, 1.0])
def test_prefill_protocol_holds_under_random_schedules(n, n_strip, p_rescale):
    if n_strip and n < 2:
        pytest.skip("a sink strip is always followed by window tiles")
    for seed in range(60):
        rng = random.Random(1000 * seed + n)
        rescale = {(w, i): rng.random() < p_rescale for w in range(4) for i in range(n)}
        run(prefill_roles(n, n_strip, rescale), seed, end_idle=True)


@pytest.mark.parametrize("mutation,error", [
    ("no_pv_wait_before_qk", r"before P V"),
    ("no_k_empty_wait", r"before Q K\^T"),
    ("one_p_barrier", r"wrong phase|two phases|in rows of warp"),
])
def test_prefill_model_catches_planted_mistakes(mutation, error):
    """Without the wait for P V two tiles back, Q K^T overwrites P before it is read;
    without the K stage's release, the next copy lands on a tile still to be used;
    with one P barrier for both parities, a wait can see a phase two tiles old."""
    caught = 0
    for seed in range(200):
        rescale = {(w, i): False for w in range(4) for i in range(6)}
        try:
            run(prefill_roles(6, 0, rescale, mutate=mutation), seed, end_idle=True)
        except ProtocolError as e:
            assert re.search(error, str(e)), str(e)
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------------------- decode


def decode_roles(units, stages, n_warps, fused, qslots=2, mutate=None):
    """One decode split block.  units: per unit of this block's share, (tiles, new_tile)
    with new_tile the tile holding the token's new row when this block writes it (the
    decode step), else None."""
    B = Barrier
    full = [B(f"full{s}", 1) for s in range(stages)]
    empty = [B(f"empty{s}", n_warps) for s in range(stages)]
    q_full = [B(f"q_full{s}", 1) for s in range(qslots)]
    q_empty = [B(f"q_empty{s}", n_warps) for s in range(qslots)]
    new_bar = B("new_bar", 1)
    st = {"stage": [None] * stages, "reads": {}, "row": {}, "q": [None] * qslots, "q_reads": {}}

    def fail(msg):
        raise ProtocolError(msg)

    def producer():
        t = 0
        token_written = not fused
        for u, (tiles, new_tile) in enumerate(units):
            for tile in range(tiles):
                if not token_written and new_tile == tile and mutate != "no_new_bar_wait":
                    yield ("wait", new_bar, 0)
                    token_written = True
                s, k = t % stages, t // stages - 1
                if k >= 0:
                    yield ("wait", empty[s], k)

                def issue(t=t, s=s, u=u, tile=tile, new_tile=new_tile):
                    prev = t - stages
                    if prev >= 0 and st["reads"].get(prev, 0) < n_warps:
                        fail(f"tile {t} copied over tile {prev} before every consumer read it")
                    if fused and new_tile == tile and st["row"].get(u) != "new":
                        fail(f"unit {u}'s tile {tile} copied before the token's row was written")
                yield ("do", issue)
                yield ("expect", full[s], 1)
                yield ("tma", full[s], 1, lambda s=s, t=t: st["stage"].__setitem__(s, t))
                t += 1
        for _ in range(stages):   # drain: every issued stage released before the block exits
            s, k = t % stages, t // stages - 1
            if k >= 0:
                yield ("wait", empty[s], k)
            t += 1

    def consumer(c):
        t, uk = 0, 0
        for u, (tiles, _) in enumerate(units):
            if fused:
                slot = uk % qslots
                yield ("wait", q_full[slot], uk // qslots)

                def read_q(u=u, slot=slot):
                    if st["q"][slot] != u:
                        fail(f"consumer {c} read q {st['q'][slot]} for unit {u}")
                    st["q_reads"][u] = st["q_reads"].get(u, 0) + 1
                yield ("do", read_q)
                yield ("arrive", q_empty[slot])
                uk += 1
            for _ in range(tiles):
                s = t % stages
                yield ("wait", full[s], t // stages)
                if mutate == "release_before_read":
                    yield ("arrive", empty[s])

                def read(t=t, s=s):
                    if st["stage"][s] != t:
                        fail(f"consumer {c} read stage {s} holding tile {st['stage'][s]} for tile {t}")
                    st["reads"][t] = st["reads"].get(t, 0) + 1
                yield ("do", read)
                if mutate != "release_before_read":
                    yield ("arrive", empty[s])
                t += 1

    def token_warp():
        # the first unit's q rows and token rows in one round, q slot 0 released
        def first():
            st["q"][0] = 0
            if units[0][1] is not None:
                st["row"][0] = "new"
        yield ("do", first)
        yield ("arrive", q_full[0])
        for u in range(1, len(units)):
            if units[u][1] is not None:
                yield ("do", lambda u=u: st["row"].__setitem__(u, "new"))
        yield ("arrive", new_bar)   # after fence.proxy.async: the copies may read the rows
        for k in range(1, len(units)):
            slot = k % qslots
            if k >= qslots:
                yield ("wait", q_empty[slot], k // qslots - 1)

            def write_q(k=k, slot=slot):
                if k >= qslots and st["q_reads"].get(k - qslots, 0) < n_warps:
                    fail(f"q of unit {k} written over unit {k - qslots}'s before every consumer read it")
                st["q"][slot] = k
            yield ("do", write_q)
            yield ("arrive", q_full[slot])

    roles = {"producer": producer()}
    for c in range(n_warps):
        roles[f"consumer{c}"] = consumer(c)
    if fused:
        roles["token"] = token_warp()
    return roles


def _random_units(rng, fused):
    units = []
    for u in range(rng.randint(1, 5)):
        tiles = rng.randint(1, 7)
        new_tile = rng.randrange(tiles) if fused and rng.random() < 0.7 else None
        units.append((tiles, new_tile))
    return units


@pytest.mark.parametrize("stages,n_warps", [(2, 2), (3, 4), (5, 3)])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_protocol_holds_under_random_schedules(stages, n_warps, fused):
    for seed in range(150):
        rng = random.Random(seed)
        run(decode_roles(_random_units(rng, fused), stages, n_warps, fused), seed, end_idle=True)


@pytest.mark.parametrize("mutation,fused,error", [
    ("release_before_read", False, r"holding tile|before every consumer read it"),
    ("no_new_bar_wait", True, r"before the token's row"),
])
def test_decode_model_catches_planted_mistakes(mutation, fused, error):
    """A consumer that releases its stage before reading it lets the next copy land
    first; a producer that does not wait for the token warp copies a tile before the
    new row is in it."""
    caught = 0
    for seed in range(300):
        rng = random.Random(seed)
        units = [(rng.randint(2, 6), 0 if fused else None) for _ in range(3)]
        try:
            run(decode_roles(units, 2, 2, fused, mutate=mutation), seed, end_idle=True)
        except ProtocolError as e:
            assert re.search(error, str(e)), str(e)
            caught += 1
    assert caught > 0


def test_a_missing_arrival_is_a_deadlock():
    """The model reports a wait that nothing will satisfy (the kernels turn it into a
    bounded wait and an error bit)."""
    roles = prefill_roles(3, 0, {(w, i): False for w in range(4) for i in range(3)})
    roles["softmax3"] = iter([])        # one softmax warp never arrives on P
    with pytest.raises(Deadlock):
        run(roles, 0, end_idle=True)
