"""Random-schedule models of the kernels' barrier protocols (test infrastructure).

Each model restates, as sequential Python programs, what the roles of one CTA
of a kernel do with their mbarriers -- the TMA producer, the single MMA
issuer, the row (softmax) warps -- and runs them under a random scheduler,
together with the two asynchronous engines: TMA copies land in any order,
tcgen05 products and commits complete in issue order.  Every shared-memory
buffer and TMEM region carries a label of what it holds; a product or a row
warp that reads a buffer checks the label it expects.  A run fails on

- an arrival beyond a barrier's count within one phase (undefined on the
  hardware),
- a read of the wrong contents (a load landed too early or too late, or a
  region was overwritten before it was read), or
- a deadlock (no role can proceed).

The barrier model follows mbarrier semantics: a phase completes when its
pending arrivals reach zero and its transaction count is zero;
try_wait.parity(P) succeeds when the current phase's parity differs from P.
The 128 row threads that arrive on a barrier together are one arrival here.
These models describe the protocols as written in prefill_tc.cu and
decode.cu; a change to a protocol there belongs here too.
"""
import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase, self.tx = name, count, count, 0, 0

    def arrive(self, tx=0, who=""):
        self.tx += tx
        self.pending -= 1
        if self.pending < 0:
            raise RuntimeError(f"{self.name}: too many arrivals in phase {self.phase} ({who})")
        self._maybe()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe()

    def _maybe(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def _schedule(rnd, actors, fifo, tma, on_mma, on_land, max_steps=200000):
    """Run the role generators (each yields ("wait", bar, parity) or
    ("step",)) with the tensor-core queue `fifo` and the in-flight copies
    `tma` until all end."""
    waiting = {k: None for k in actors}
    alive = set(actors)
    steps = 0
    while alive or fifo or tma:
        steps += 1
        if steps > max_steps:
            raise RuntimeError("no progress")
        choices = [("role", a) for a in sorted(alive)
                   if waiting[a] is None or waiting[a][1].done(waiting[a][2])]
        if fifo:
            choices.append(("tc", None))
        if tma:
            choices.append(("tma", None))
        if not choices:
            raise RuntimeError("deadlock: " + ", ".join(
                f"{a} on {w[1].name}/{w[2]}" for a, w in waiting.items() if a in alive and w))
        kind, a = rnd.choice(choices)
        if kind == "role":
            try:
                w = next(actors[a])
                # ("step",): a point where other actors may run in between
                waiting[a] = None if w[0] == "step" else w
            except StopIteration:
                alive.discard(a)
                waiting[a] = None
        elif kind == "tc":
            op = fifo.pop(0)
            if op[0] == "commit":
                op[1].arrive(who="commit")
            else:
                on_mma(op)
        else:
            on_land(tma.pop(rnd.randrange(len(tma))))


def multi_block_prefill(units, seed, kst=2, shared_k0_barrier=False):
    """Prefill units of several key blocks (global layers, wide windows):
    `units` lists each unit's block count.  K in kst stages, V in one; K_0 of
    a unit on the K_0 barrier of its stage (or, planted mistake, on one
    barrier for all units), V_j and K_{j+1} on tile A's P barrier, the K
    stages released by tile B's rows."""
    rnd = random.Random(seed)
    k0_full = [Bar(f"k0_full{i}", 1) for i in range(1 if shared_k0_barrier else kst)]
    pf = [Bar("p_full0", 3), Bar("p_full1", 1)]  # tile A: rows + V_j + (K_{j+1} or stand-in)
    kv_empty = [Bar(f"kv_empty{i}", 1) for i in range(kst + 1)]
    q_full = [Bar(f"q_full{t}", 1) for t in range(2)]
    q_ready = [Bar(f"q_ready{t}", 1) for t in range(2)]
    q_empty = [Bar(f"q_empty{t}", 1) for t in range(2)]
    s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
    pv_done = [Bar(f"pv_done{t}", 1) for t in range(2)]
    o_free = [Bar(f"o_free{t}", 1) for t in range(2)]
    slot, tm, tma, fifo = {}, {}, [], []

    def producer():
        kq = vq = 0
        qf = [0, 0]

        def load_k(n, j, first):
            nonlocal kq
            st = kq % kst
            yield ("wait", kv_empty[st], ((kq // kst) & 1) ^ 1)
            if not first and vq > 0:
                yield ("wait", pf[0], (vq - 1) & 1)
            b = k0_full[0 if shared_k0_barrier else st] if first else pf[0]
            b.arrive(tx=1, who="producer K")
            tma.append((("K", st), ("K", n, j), b))
            kq += 1

        for n, nb in enumerate(units):
            # the CTA's first unit loads its Q tiles before K_0
            if n > 0:
                yield from load_k(n, 0, True)
            for t in range(2):
                yield ("wait", q_empty[t], (qf[t] & 1) ^ 1)
                q_full[t].arrive(tx=1, who="producer Q")
                tma.append((("Q", t), ("Qraw", n, t), q_full[t]))
                qf[t] += 1
            if n == 0:
                yield from load_k(n, 0, True)
            for j in range(nb):
                if j + 1 < nb:
                    yield from load_k(n, j + 1, False)
                yield ("wait", kv_empty[kst], (vq & 1) ^ 1)
                pf[0].arrive(tx=1, who="producer V")
                tma.append((("V",), ("V", n, j), pf[0]))
                vq += 1

    def mma():
        uc = kc = blk = 0
        k0c = [0] * len(k0_full)
        for n, nb in enumerate(units):
            k0 = kc % kst
            kc += 1
            bi = 0 if shared_k0_barrier else k0
            yield ("wait", k0_full[bi], (uc if shared_k0_barrier else k0c[bi]) & 1)
            k0c[bi] += 1
            for t in range(2):
                yield ("wait", q_ready[t], uc & 1)
                fifo.append(("mma", {("Q", t): ("Qrot", n, t), ("K", k0): ("K", n, 0)},
                             {("S", t): ("S", n, 0)}))
                fifo.append(("commit", s_full[t]))
                if nb == 1:
                    fifo.append(("commit", q_empty[t]))
            for j in range(nb):
                more = j + 1 < nb
                kn = None
                for t in range(2):
                    yield ("wait", pf[t], blk & 1)
                    if j == 0 and uc > 0:
                        yield ("wait", o_free[t], (uc - 1) & 1)
                    fifo.append(("mma", {("S", t): ("P", n, j), ("V",): ("V", n, j)},
                                 {("O", t): ("O", n, j)}))
                    if not more:
                        fifo.append(("commit", pv_done[t]))
                    if t == 1:
                        fifo.append(("commit", kv_empty[kst]))
                    if more:
                        if t == 0:
                            kn = kc % kst
                            kc += 1
                        fifo.append(("mma", {("Q", t): ("Qrot", n, t), ("K", kn): ("K", n, j + 1)},
                                     {("S", t): ("S", n, j + 1)}))
                        fifo.append(("commit", s_full[t]))
                        if j + 2 == nb:
                            fifo.append(("commit", q_empty[t]))
                blk += 1
            uc += 1

    def rows(t):
        uc = blk = 0
        prev = None

        def epilogue(pn, pnb):
            yield ("wait", pv_done[t], pn & 1)
            assert tm.get(("O", t)) == ("O", pn, pnb - 1), f"epilogue of tile {t} read {tm.get(('O', t))}"
            o_free[t].arrive(who=f"rows {t} o_free")

        for n, nb in enumerate(units):
            yield ("wait", q_full[t], uc & 1)
            assert slot.get(("Q", t)) == ("Qraw", n, t), f"RoPE of tile {t} read {slot.get(('Q', t))}"
            slot[("Q", t)] = ("Qrot", n, t)
            q_ready[t].arrive(who=f"rows {t} q_ready")
            if prev is not None:
                yield from epilogue(*prev)
            for j in range(nb):
                yield ("wait", s_full[t], blk & 1)
                if t == 1:
                    kv_empty[blk % kst].arrive(who="rows 1 K release")
                assert tm.get(("S", t)) == ("S", n, j), f"softmax of tile {t} read {tm.get(('S', t))}"
                tm[("S", t)] = ("P", n, j)
                pf[t].arrive(who=f"rows {t} P")
                if t == 0 and j + 1 == nb:
                    pf[0].arrive(who="rows 0 stand-in")
                blk += 1
            prev = (uc, nb)
            uc += 1
        if prev is not None:
            yield from epilogue(*prev)

    def on_mma(op):
        for key, lab in op[1].items():
            cur = slot.get(key) if key[0] in ("Q", "K", "V") else tm.get(key)
            if cur != lab:
                raise RuntimeError(f"product reads {key}: holds {cur}, expects {lab}")
        for key, lab in op[2].items():
            if key[0] == "O" and lab[2] > 0 and tm.get(key) != ("O", lab[1], lab[2] - 1):
                raise RuntimeError(f"PV accumulates onto {tm.get(key)}, expects block {lab[2] - 1}")
            tm[key] = lab

    def on_land(copy):
        key, lab, b = copy
        slot[key] = lab
        b.complete_tx(1)

    _schedule(rnd, {"producer": producer(), "mma": mma(), "rows0": rows(0), "rows1": rows(1)},
              fifo, tma, on_mma, on_land)


def one_block_prefill(nunits, seed, stage_a_after_own_pv=False, v_without_o_read=False):
    """Window units whose key band is one block: Q_t, K and V are released
    through the phases of S_t, S_B and PV_B; O_t sits over S_t's upper TMEM
    columns, so the next S_t waits until the epilogue has read O_t.  Tile A's
    epilogue stages O in the V stage once PV_B of the unit is done, and the
    next V block loads once that staging has been read (o_read).  Planted
    mistakes: tile A staging after its own PV only; V loaded without o_read."""
    rnd = random.Random(seed)
    q_full = [Bar(f"q_full{t}", 1) for t in range(2)]
    q_ready = [Bar(f"q_ready{t}", 1) for t in range(2)]
    s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
    p_full = [Bar(f"p_full{t}", 1) for t in range(2)]
    pv_done = [Bar(f"pv_done{t}", 1) for t in range(2)]
    o_free = [Bar(f"o_free{t}", 1) for t in range(2)]
    kv_full = [Bar("kv_full0", 1), Bar("kv_full1", 1)]
    o_read = Bar("o_read", 1)
    smem, tm, tma, fifo = {}, {}, [], []
    pv_ran = {}  # (tile, unit) -> True once that PV has executed

    def producer():
        qf = [0, 0]
        for n in range(nunits):
            for t in range(2):
                if qf[t] > 0:
                    yield ("wait", s_full[t], (qf[t] - 1) & 1)
                q_full[t].arrive(tx=1)
                tma.append((("Q", t), ("Qraw", n), q_full[t]))
                qf[t] += 1
            if n > 0:
                yield ("wait", s_full[1], (n - 1) & 1)
            kv_full[0].arrive(tx=1)
            tma.append((("K",), ("K", n), kv_full[0]))
            if n > 0:
                yield ("wait", pv_done[1], (n - 1) & 1)
                if not v_without_o_read:
                    yield ("wait", o_read, (n - 1) & 1)
            kv_full[1].arrive(tx=1)
            tma.append((("V",), ("V", n), kv_full[1]))

    def mma():
        for uc in range(nunits):
            yield ("wait", kv_full[0], uc & 1)
            for t in range(2):
                yield ("wait", q_ready[t], uc & 1)
                if uc > 0:
                    yield ("wait", o_free[t], (uc - 1) & 1)
                fifo.append(("qk", t, uc))
                fifo.append(("commit", s_full[t]))
            yield ("wait", kv_full[1], uc & 1)
            for t in range(2):
                yield ("wait", p_full[t], uc & 1)
                fifo.append(("pv", t, uc))
                fifo.append(("commit", pv_done[t]))

    def rows(t):
        prev = None
        for n in range(nunits):
            yield ("wait", q_full[t], n & 1)
            assert smem.get(("Q", t)) == ("Qraw", n), f"RoPE of tile {t} read {smem.get(('Q', t))}"
            smem[("Q", t)] = ("Qrot", n)
            q_ready[t].arrive()
            if prev is not None:
                yield from epilogue(t, prev)
            yield ("wait", s_full[t], n & 1)
            assert tm.get(("lo", t)) == ("S", n), f"softmax read {tm.get(('lo', t))}"
            tm[("lo", t)] = ("P", n)
            p_full[t].arrive()
            prev = n
        if prev is not None:
            yield from epilogue(t, prev)

    def epilogue(t, n):
        yield ("wait", pv_done[t], n & 1)
        assert tm.get(("up", t)) == ("O", n), f"epilogue read {tm.get(('up', t))}"
        tm[("up", t)] = ("Oread", n)
        o_free[t].arrive()
        if t == 0:
            # stage into the V stage; the TMA stores read it out, then o_read
            if not stage_a_after_own_pv:
                yield ("wait", pv_done[1], n & 1)
            if not pv_ran.get((1, n)):
                raise RuntimeError(f"tile A stages O of unit {n} over V while PV_B still reads it")
            smem[("V",)] = ("staged", n)
            yield ("step",)
            if smem.get(("V",)) != ("staged", n):
                raise RuntimeError(f"V block landed over tile A's staged O of unit {n}")
            o_read.arrive()

    def on_mma(op):
        _, t, n = op
        if op[0] == "qk":
            if smem.get(("Q", t)) != ("Qrot", n) or smem.get(("K",)) != ("K", n):
                raise RuntimeError(f"S_{t} of unit {n} reads Q {smem.get(('Q', t))}, K {smem.get(('K',))}")
            if n > 0 and tm.get(("up", t)) != ("Oread", n - 1):
                raise RuntimeError(f"S_{t} of unit {n} overwrites O before its epilogue read it")
            tm[("lo", t)] = ("S", n)
            tm[("up", t)] = ("S", n)
        else:
            if tm.get(("lo", t)) != ("P", n) or smem.get(("V",)) != ("V", n):
                raise RuntimeError(f"PV_{t} of unit {n} reads P {tm.get(('lo', t))}, V {smem.get(('V',))}")
            tm[("up", t)] = ("O", n)
            pv_ran[(t, n)] = True

    def on_land(copy):
        key, lab, b = copy
        smem[key] = lab
        b.complete_tx(1)

    _schedule(rnd, {"producer": producer(), "mma": mma(), "rows0": rows(0), "rows1": rows(1)},
              fifo, tma, on_mma, on_land)


def split_kv_decode(items, seed, nst=5, epilogue_on_pv_done=False):
    """The split-KV decode kernel: `items` lists each item's block count.
    K/V blocks stream through nst stages, each released by a row thread once
    it has seen S of the block two later; the epilogue waits on the per-item
    barrier o_done (or, planted mistake, on pv_done's parity, which can
    alias there); a rescale of O waits on pv_done for the previous block."""
    rnd = random.Random(seed)
    full = [Bar(f"full{i}", 1) for i in range(nst)]
    empty = [Bar(f"empty{i}", 1) for i in range(nst)]
    q_ready = [Bar(f"q_ready{i}", 1) for i in range(2)]
    q_empty = [Bar(f"q_empty{i}", 1) for i in range(2)]
    s_full = [Bar(f"s_full{i}", 1) for i in range(2)]
    p_full = [Bar(f"p_full{i}", 1) for i in range(2)]
    pv_done, o_done, o_free = Bar("pv_done", 1), Bar("o_done", 1), Bar("o_free", 1)
    stage, tm, q, tma, fifo = {}, {}, {}, [], []

    def producer():
        pos = 0
        for nb in items:
            for _ in range(nb):
                st = pos % nst
                yield ("wait", empty[st], ((pos // nst) & 1) ^ 1)
                full[st].arrive(tx=1, who="producer")
                tma.append((st, ("KV", pos), full[st]))
                pos += 1

    def mma():
        qc = qk = done = 0
        owner = {}

        def issue_qk(qb, g):
            st = g % nst
            yield ("wait", full[st], (g // nst) & 1)
            fifo.append(("mma", [("st", st, g), ("q", qb, owner[qb])], ("S", g & 1), ("S", g)))
            fifo.append(("commit", s_full[g & 1]))

        for it, nb in enumerate(items):
            qb = qc & 1
            yield ("wait", q_ready[qb], (qc >> 1) & 1)
            qc += 1
            owner[qb] = it
            b0 = qk
            yield from issue_qk(qb, qk)
            qk += 1
            if nb == 1:
                fifo.append(("commit", q_empty[qb]))
            for j in range(nb):
                if j + 1 < nb:
                    yield from issue_qk(qb, qk)
                    qk += 1
                    if j + 2 == nb:
                        fifo.append(("commit", q_empty[qb]))
                g = b0 + j
                yield ("wait", p_full[g & 1], (g >> 1) & 1)
                if j == 0 and done > 0:
                    yield ("wait", o_free, (done - 1) & 1)
                fifo.append(("mma", [("st", g % nst, g), ("P", g & 1, g)], ("O", 0), ("O", it, j)))
                fifo.append(("commit", pv_done))
                if j + 1 == nb:
                    fifo.append(("commit", o_done))
            done += 1

    def rows():
        qc = blk = ni = 0
        prev = None

        def epilogue():
            if epilogue_on_pv_done:
                yield ("wait", pv_done, (blk - 1) & 1)
            else:
                yield ("wait", o_done, (ni - 1) & 1)
            assert tm.get(("O", 0)) == ("O", prev[0], prev[1] - 1), \
                f"epilogue of item {prev[0]} read {tm.get(('O', 0))}"

        for it, nb in enumerate(items):
            qb = qc & 1
            yield ("wait", q_empty[qb], ((qc >> 1) & 1) ^ 1)
            qc += 1
            q[qb] = it
            q_ready[qb].arrive(who="rows q_ready")
            if prev is not None:
                yield from epilogue()
                o_free.arrive(who="rows o_free")
            for j in range(nb):
                yield ("wait", s_full[blk & 1], (blk >> 1) & 1)
                if blk >= 2:
                    empty[(blk - 2) % nst].arrive(who="rows stage release")
                assert tm.get(("S", blk & 1)) == ("S", blk), f"softmax of block {blk} read {tm.get(('S', blk & 1))}"
                # the V rows of a partial block are zeroed in the block's stage
                assert stage.get(blk % nst) == ("KV", blk), f"V rows of block {blk}: stage holds {stage.get(blk % nst)}"
                if j > 0 and rnd.random() < 0.25:  # a rescale of O
                    yield ("wait", pv_done, (blk - 1) & 1)
                    assert tm.get(("O", 0)) == ("O", it, j - 1), f"rescale read {tm.get(('O', 0))}"
                tm[("S", blk & 1)] = ("P", blk)
                p_full[blk & 1].arrive(who="rows P")
                blk += 1
            prev = (it, nb)
            ni += 1
        if prev is not None:
            yield from epilogue()

    def on_mma(op):
        for r in op[1]:
            if r[0] == "st":
                if stage.get(r[1]) != ("KV", r[2]):
                    raise RuntimeError(f"product reads stage {r[1]}: {stage.get(r[1])}, expects block {r[2]}")
            elif r[0] == "q":
                if q.get(r[1]) != r[2]:
                    raise RuntimeError(f"QK reads Q buffer {r[1]}: item {q.get(r[1])}, expects {r[2]}")
            elif tm.get(("S", r[1])) != ("P", r[2]):
                raise RuntimeError(f"PV reads {tm.get(('S', r[1]))}, expects P of block {r[2]}")
        lab = op[3]
        if op[2][0] == "O" and lab[2] > 0 and tm.get(op[2]) != ("O", lab[1], lab[2] - 1):
            raise RuntimeError(f"PV accumulates onto {tm.get(op[2])}, expects {lab}")
        tm[op[2]] = lab

    def on_land(copy):
        st, lab, b = copy
        stage[st] = lab
        b.complete_tx(1)

    _schedule(rnd, {"producer": producer(), "mma": mma(), "rows": rows()}, fifo, tma, on_mma, on_land)


def unit_queue(entries, readers, seed, nq=4, skip_empty_wait=False):
    """The prefill's unit queue: the producer publishes `entries` unit indices
    (then the end, -1) into nq slots, each with a full barrier (count 1) and
    an empty barrier (one arrival per reader); every reader takes the entries
    in order at its own pace -- the MMA issuer one per unit, the softmax warps
    of one-block units one entry ahead of the unit they work on.  Planted
    mistake: a producer that reuses a slot without its empty barrier."""
    rnd = random.Random(seed)
    full = [Bar(f"unit_full{q}", 1) for q in range(nq)]
    empty = [Bar(f"unit_empty{q}", readers) for q in range(nq)]
    slot = {}
    seq = list(range(entries)) + [-1]

    def producer():
        for pn, u in enumerate(seq):
            q = pn % nq
            if pn >= nq and not skip_empty_wait:
                yield ("wait", empty[q], ((pn // nq) & 1) ^ 1)
            slot[q] = u
            full[q].arrive()
            yield ("step",)

    def reader(i):
        for n, want in enumerate(seq):
            q = n % nq
            yield ("wait", full[q], (n // nq) & 1)
            if slot.get(q) != want:
                raise RuntimeError(f"reader {i} took {slot.get(q)} as entry {n}, not {want}")
            empty[q].arrive()
            for _ in range(rnd.randint(0, 3)):  # its own work between entries
                yield ("step",)

    actors = {"producer": producer()}
    actors.update({f"reader{i}": reader(i) for i in range(readers)})
    _schedule(rnd, actors, [], [], None, None)
