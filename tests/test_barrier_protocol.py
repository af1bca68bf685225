"""Model check of the attention kernel's mbarrier schedule (CPU, no GPU).

The kernel's roles (two TMA streams -- q tiles and K, and V -- or, for
token-granular pages, a q-tile stream and row-gather warps; an optional FP8
dequant warpgroup; the tcgen05 issuer; one softmax warpgroup per q-tile slot
of 4 warps) synchronise through
mbarriers waited on by phase parity.  This test replays that schedule -- the
same waits, arrivals and commits, in the same order per role as
csrc/bip_attn_impl.cuh -- with random completion delays for TMA loads and MMAs and
random interleavings of the roles, for every kernel variant, and checks two
properties on many schedules:

* no deadlock: every role finishes;
* no aliased wait: when a parity wait returns, the barrier has completed
  exactly the phase waited for (not one fewer, not two more).  A barrier that
  can run two phases ahead of its waiter reads as "not yet" forever; one that
  a waiter can read before its phase completes lets it consume data early.

tcgen05.commit arrives once every MMA issued before it by the same thread has
completed (modelled as in-order completion of the issuer's operations).
"""

import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "over-arrival"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def _simulate(NT, NS, ST, SS, items, seed, warps=4, GW=0, DQ=1, HP=False):
    """items: list of (nb, mask); SS > 0 models FP8 staging + dequant (DQ
    dequant warpgroups taking alternate blocks); HP models the early first
    half of P (P_HALF: the issuer starts the PV of the first 64 keys, then
    waits P_FULL for the rest; a warp that rescales O publishes its half only
    at the end of the block); GW > 0
    models token-granular pages: GW row-gather warps per stream, whose 32
    lanes each arrive on the landing barrier when their own copies land,
    and a q/K producer that loads q tiles only."""
    rnd = random.Random(seed)
    B = {}

    def bar(name, count=1):
        B.setdefault(name, _Bar(count))

    land = 32 * GW if GW else 1
    for s in range(ST):
        for n in ("K_FULL", "V_FULL"):
            bar(f"{n}{s}", 128 if SS else land)
        bar(f"K_FREE{s}"), bar(f"V_FREE{s}")
    for s in range(SS):
        bar(f"K8_FULL{s}", land), bar(f"V8_FULL{s}", land), bar(f"K8_FREE{s}", 128), bar(f"V8_FREE{s}", 128)
    for t in range(NT):
        for s in range(NS):
            bar(f"S_FULL{t}{s}"), bar(f"P_FULL{t}{s}", 32 * warps), bar(f"O_DONE{t}{s}")
            bar(f"P_HALF{t}{s}", 32 * warps)
    bar("Q_FULL"), bar("Q_FREE"), bar("V_TX")
    bar("Q_READY", 128), bar("QS_FREE", 32 * warps * NT)  # FP8: q tile converted / its row scales read
    clock, pending, last_mma = [0], [], [0]

    def later(name, lo=1, hi=8):
        pending.append((clock[0] + rnd.randint(lo, hi), name))

    def gatherer(is_v):
        """One row-gather warp: the same block schedule as the TMA producer;
        each lane's copies land after their own delay, then that lane
        arrives."""
        ring = SS if SS else ST
        kv = ("V8" if SS else "V") if is_v else ("K8" if SS else "K")
        b = 0
        for nb, _ in items:
            for _ in range(nb):
                slot, use = b % ring, b // ring
                if use > 0:
                    yield wait(f"{kv}_FREE{slot}", use - 1)
                for _ in range(32):
                    later(f"{kv}_FULL{slot}", 1, 12)
                b += 1
                yield None

    def q_loader():
        for n in range(len(items)):
            if n > 0:
                yield wait("Q_FREE", n - 1)
            later("Q_FULL")
            yield None

    def commit(name):
        last_mma[0] = max(last_mma[0], clock[0]) + rnd.randint(1, 5)
        pending.append((last_mma[0], name))

    def wait(name, idx):
        return ("wait", name, idx)

    def producer(is_v):
        """One warp streams the q tiles and K, another streams V; an item's
        first ring-depth K blocks go out before its q tiles.  A bf16 V block
        that ends past kv_len (here: every item's last block) lands on V_TX;
        the V warp waits for it, zeroes the tail and completes V_FULL."""
        ring = SS if SS else ST
        kv = ("V8" if SS else "V") if is_v else ("K8" if SS else "K")
        b, n_tail = 0, 0
        for n, (nb, mask) in enumerate(items):
            q_done = is_v

            def load_q():
                if n > 0:
                    yield wait("Q_FREE", n - 1)
                later("Q_FULL")

            for j in range(nb):
                if not q_done and j == min(ring, nb):
                    yield from load_q()
                    q_done = True
                slot, use = b % ring, b // ring
                if use > 0:
                    yield wait(f"{kv}_FREE{slot}", use - 1)
                if is_v and not SS and j == nb - 1:
                    later("V_TX")
                    yield wait("V_TX", n_tail)
                    n_tail += 1
                    B[f"V_FULL{slot}"].arrive()
                else:
                    later(f"{kv}_FULL{slot}")
                b += 1
                yield None
            if not q_done:
                yield from load_q()

    def dequant(wg=0, nwg=1):
        """Warpgroup 0 converts each item's q tile (after the softmax read the
        previous tile's row scales); with two warpgroups wg 0 dequantizes
        every K block and wg 1 every V block, with one it does K then V:
        staged codes into registers, stage freed, ring slot taken."""
        b = 0
        for n, (nb, _) in enumerate(items):
            if wg == 0:
                if n > 0:
                    yield wait("QS_FREE", n - 1)
                yield wait("Q_FULL", n)
                for _ in range(128):
                    B["Q_READY"].arrive()
            for _ in range(nb):
                ss, slot = b % SS, b % ST
                for kv in (("K", "V")[wg],) if nwg == 2 else ("K", "V"):
                    yield wait(f"{kv}8_FULL{ss}", b // SS)
                    for _ in range(128):  # codes in registers: the stage is free
                        B[f"{kv}8_FREE{ss}"].arrive()
                    if b // ST > 0:
                        yield wait(f"{kv}_FREE{slot}", b // ST - 1)
                    for _ in range(128):
                        B[f"{kv}_FULL{slot}"].arrive()
                b += 1
                yield None

    def issuer():
        gb, s_cnt, pv_cnt, k_seen = 0, [0] * NT, [0] * NT, [0]
        for n, (nb, mask) in enumerate(items):
            yield wait("Q_READY" if SS else "Q_FULL", n)
            last = max(t for t in range(NT) if mask >> t & 1)
            if NT == 1:  # q tile copied into TMEM once the previous item's last S has completed
                if n > 0:
                    yield wait(f"S_FULL0{(s_cnt[0] - 1) % NS}", (s_cnt[0] - 1) // NS)
                commit("Q_FREE")

            def issue_s(t, j):
                kb = gb + j
                if kb >= k_seen[0]:  # another slot's S may already have seen it land
                    yield wait(f"K_FULL{kb % ST}", kb // ST)
                    k_seen[0] = kb + 1
                commit(f"S_FULL{t}{s_cnt[t] % NS}")
                if t == last:
                    commit(f"K_FREE{kb % ST}")
                    if NT == 2 and j == nb - 1:
                        commit("Q_FREE")
                s_cnt[t] += 1

            for j in range(min(NS, nb)):
                for t in range(NT):
                    if mask >> t & 1:
                        yield from issue_s(t, j)
            for j in range(nb):
                vb = gb + j
                vready = False
                for t in range(NT):
                    if not mask >> t & 1:
                        continue
                    yield wait(f"{'P_HALF' if HP else 'P_FULL'}{t}{pv_cnt[t] % NS}", pv_cnt[t] // NS)
                    if not vready:
                        yield wait(f"V_FULL{vb % ST}", vb // ST)
                        vready = True
                    if HP:  # the first 64 keys' PV is queued; the rest needs all of P
                        yield wait(f"P_FULL{t}{pv_cnt[t] % NS}", pv_cnt[t] // NS)
                    commit(f"O_DONE{t}{pv_cnt[t] % NS}")
                    pv_cnt[t] += 1
                    if j + NS < nb:
                        yield from issue_s(t, j + NS)
                commit(f"V_FREE{vb % ST}")
                yield None
            gb += nb

    def softmax(t):
        cnt, pv_seen = 0, 0

        def wait_pv(x):
            nonlocal pv_seen
            if pv_seen <= x:
                yield wait(f"O_DONE{t}{x % NS}", x // NS)
                pv_seen = x + 1

        for n, (nb, mask) in enumerate(items):
            if SS:  # FP8: the tile's row scales, read once the tile is converted
                yield wait("Q_READY", n)
                for _ in range(32):
                    B["QS_FREE"].arrive()
            if not mask >> t & 1:
                continue
            for blk in range(nb):
                yield wait(f"S_FULL{t}{cnt % NS}", cnt // NS)
                rescale = blk > 0 and rnd.random() < 0.3            # a row's max moved: rescale O
                if HP and not rescale:                               # first half of P out early
                    for _ in range(32):
                        B[f"P_HALF{t}{cnt % NS}"].arrive()
                    yield None
                if rescale and NS == 2:
                    yield from wait_pv(cnt - 1)
                if HP and rescale:
                    for _ in range(32):
                        B[f"P_HALF{t}{cnt % NS}"].arrive()
                for _ in range(32):
                    B[f"P_FULL{t}{cnt % NS}"].arrive()
                cnt += 1
                yield None
            yield from wait_pv(cnt - 1)                            # segment end: read O
            for _ in range(rnd.randint(0, 40)):                    # a slow epilogue lets other roles run ahead
                yield None

    if GW:
        roles = [("q_loader", q_loader()), ("issuer", issuer())]
        roles += [(f"gather_{kv}{w}", gatherer(kv == "v")) for kv in "kv" for w in range(GW)]
    else:
        roles = [("producer_k", producer(False)), ("producer_v", producer(True)), ("issuer", issuer())]
    roles += [(f"softmax{t}.{w}", softmax(t)) for t in range(NT) for w in range(warps)]
    if SS:
        roles += [(f"dequant{w}", dequant(w, DQ)) for w in range(DQ)]
    state, done = {n: None for n, _ in roles}, set()
    for _ in range(500000):
        clock[0] += 1
        pending.sort()
        while pending and pending[0][0] <= clock[0]:
            B[pending.pop(0)[1]].arrive()
        order = list(roles)
        rnd.shuffle(order)
        moved = False
        for name, gen in order:
            if name in done:
                continue
            st = state[name]
            if st is not None:
                _, bname, idx = st
                if not B[bname].done(idx & 1):
                    continue
                assert B[bname].phase == idx + 1, f"{name}: aliased wait on {bname} phase {idx}"
                state[name] = None
            moved = True
            try:
                state[name] = next(gen)
            except StopIteration:
                done.add(name)
        if len(done) == len(roles):
            return
        assert moved or pending, f"deadlock: {state}"
    raise AssertionError("schedule did not finish")


VARIANTS = {  # (NT slots, NS S buffers, ST ring stages, SS FP8 staging stages, GW gather warps per stream,
    #           DQ dequant warpgroups, HP early half of P: FP8 pages with 128-key blocks)
    "d128_two_tiles": (2, 1, 2, 0, 0, 1, False),
    "d128_one_tile": (1, 2, 3, 0, 0, 1, False),
    "d256": (1, 2, 2, 0, 0, 1, False),
    "d128_fp8": (1, 2, 2, 2, 0, 2, True),
    "d128_fp8_two_tiles": (2, 1, 2, 1, 0, 1, True),
    "d256_fp8": (1, 2, 2, 1, 0, 2, False),
    "d128_rows": (1, 2, 3, 0, 4, 1, False),
    "d256_rows": (1, 2, 2, 0, 4, 1, False),
    "d128_fp8_rows": (1, 2, 2, 2, 2, 1, True),
    "d256_fp8_rows": (1, 2, 2, 1, 2, 1, False),
}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_schedule_never_deadlocks_or_aliases(variant):
    NT, NS, ST, SS, GW, DQ, HP = VARIANTS[variant]
    full = (1 << NT) - 1
    item_sets = [[(1, full)], [(9, full)], [(4, full), (1, full), (17, full)], [(3, 1), (2, full), (5, 1)],
                 [(6, full), (1, full), (1, full), (2, full), (1, full), (5, full)]]  # short items run ahead
    if NT == 2:
        item_sets.append([(6, 2), (2, 1), (7, 3)])
    for items in item_sets:
        for seed in range(60 if not GW else 25):
            _simulate(NT, NS, ST, SS, items, seed, GW=GW, DQ=DQ, HP=HP)
