"""Host interpreter of the decode step's task lists: the kernel's counter
protocol run on the CPU, without a GPU.

Each SM is two agents, as in the kernel: a producer that walks the SM's task
list, resolves every task into chunks (the routing-dependent shares with the
same rules the kernel applies on the device), hands them over through a ring
of 8 task slots and streams their stages through a ring of 5; and a consumer
that takes the chunks in order, waits on global counters where the kernel
does, consumes the stages and arrives on counters where the kernel does.  An
agent runs only while its next action is possible (a counter at its target, a
free slot, a stage that has arrived); the agents are interleaved in a random
order with random run lengths, standing in for arbitrary delays.  If no agent
can move before every list has ended, the step would hang: the interpreter
reports every wait that is stuck (what the kernel's bounded waits report as a
time-out).

Wait / arrive semantics (the kernel's consumer and producer code):
  P1 / FINAL first chunk   wait OUT(l-1) >= out target (+ the bump word)
  P1 chunk ending router rows  arrive RTR(l);  P1 last chunk  arrive P1(l)
  ROUTE                    one token: the producer waits RTR(l) >= router SMs;
                           several: the consumer does, then the producer may
                           resolve this SM's UP and DOWN shares
  ATTN item                wait P1(l) >= all SMs; arrive ITEMS(l, seq)
  COMBINE                  per unit wait ITEMS(l, seq) >= its split count;
                           arrive COMB(l)
  UP last chunk            arrive UP(l)
  OUT O-proj chunk         wait COMB(l) >= combine SMs; one token: the last
                           chunk arrives OUT(l); several: a last chunk waits
                           DOWN(l) >= down SMs and arrives OUT(l)
  DOWN                     one token: the producer waits UP(l) >= UP SMs
                           before streaming the partials; the chunk arrives
                           OUT(l); several: chunks wait UP(l), the last arrives
                           DOWN(l)
Targets: P1 = SMs; OUT = SMs (+ DOWN SMs with one token); the others the SM
counts the host plan reports.  This module restates the kernel's chunking and
share rules; it shares no code with it.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field

OP_P1, OP_ROUTE, OP_ATTN, OP_UP, OP_COMBINE, OP_OUT, OP_FINAL, OP_DOWN = 1, 2, 3, 4, 5, 6, 7, 8
F_OP, F_LAYER, F_A0, F_A1, F_BUMP, F_B0, F_B1 = 0, 1, 2, 3, 5, 6, 7
STAGE_BYTES, TASK_SLOTS, STAGES = 32768, 8, 5


def rows_per_stage(K):
    return max(1, STAGE_BYTES // (2 * K))


def nseg(K):
    return 1 if K < 256 else K // 256


def chunk_rows(K, nt):
    return min(512, 2048 // (nseg(K) * max(nt, 1)))


def one_rows(K):
    return 128 if K in (2048, 4096) else 2048


def dshare(total, n, s):
    return total * s // n, total * (s + 1) // n


def cdiv(a, b):
    return -(-a // b)


@dataclass
class Chunk:
    waits: list = field(default_factory=list)      # consumer: [(counter, target)] before its stages
    stages: int = 0
    arrives: list = field(default_factory=list)    # consumer: counters +1 at its end
    pre_stage_wait: tuple | None = None            # producer: (counter, target) after hand-over
    routes: int = -1                                # several tokens ROUTE: layer routed
    end: bool = False
    # filled while running
    issued: int = 0


class Deadlock(AssertionError):
    pass


class StepSim:
    """One step of the plan from mk_plan_step for `dims`, batch and lengths;
    ``routing[l]`` = [batch][top_k] experts of layer l (drawn by the caller)."""

    def __init__(self, dims, plan, batch, routing, n_sm, claim_rows=0):
        self.d, self.plan, self.B, self.routing, self.n_sm = dims, plan, batch, routing, n_sm
        self.one = batch == 1
        # several tokens, claim_rows > 0: the expert tiles come from the
        # per-layer claim counters (taken in the interleaving's order)
        self.claim_rows = 0 if self.one else claim_rows
        self.claims = {}
        self.counters = {}
        self.route_done = [0] * n_sm
        self.coverage = {"up": {}, "down": {}}      # (layer) -> list of resolved ranges

    # ------------------------------------------------------ targets
    def target(self, kind):
        p = self.plan
        return {"p1": self.n_sm, "rtr": p["n_rtr_sms"], "up": p["n_up_sms"], "comb": p["n_comb_sms"],
                "down": p["n_down_sms"],
                "out": self.n_sm + (p["n_down_sms"] if self.one else 0)}[kind]

    def active(self, l):
        """(n_act, count per active expert) of layer l: experts ascending."""
        ex = sorted(set(int(e) for e in self.routing[l].reshape(-1)))
        cnt = [int((self.routing[l] == e).sum()) for e in ex]
        return len(ex), cnt

    # ------------------------------------------------------ producer: resolve one task into chunks
    def rows_chunks(self, lo, hi, cr, K, first, last, last_extra=None):
        out = []
        c0 = lo
        while c0 < hi:
            n = min(cr, hi - c0)
            ch = Chunk(stages=cdiv(n, rows_per_stage(K)))
            ch.first = first and c0 == lo
            ch.last = last and c0 + cr >= hi
            ch.extra = last_extra if c0 + cr >= hi else None
            ch.rows = n
            out.append(ch)
            c0 += cr
        return out

    def resolve(self, s, t):
        d = self.d
        op, l, a0, a1 = int(t[F_OP]), int(t[F_LAYER]), int(t[F_A0]), int(t[F_A1])
        H, B = d.hidden, self.B
        chunks = []
        if op in (OP_P1, OP_FINAL):
            bump = int(t[F_BUMP])
            b0, b1 = int(t[F_B0]), int(t[F_B1])
            if op == OP_FINAL:
                b0 = b1 = 0
            if self.one:
                cr = one_rows(H)
                phases = [(a0, a1, True), (b0, b1, False)]
                seq = []
                for lo, hi, is_rtr in phases:
                    c0 = lo
                    while c0 < hi:
                        c1 = min(hi, c0 + cr)
                        seq.append((c1 - c0, is_rtr and op == OP_P1 and c1 >= hi))
                        c0 = c1
                if not seq:
                    seq = [(0, False)]
                for i, (n, rtr) in enumerate(seq):
                    ch = Chunk(stages=cdiv(n, rows_per_stage(H)))
                    ch.first, ch.last, ch.extra, ch.rows = i == 0, i == len(seq) - 1, ("rtr" if rtr else None), n
                    chunks.append(ch)
            else:
                cr = chunk_rows(H, B)
                if op == OP_FINAL:
                    if a1 <= a0:
                        ch = Chunk(); ch.first, ch.last, ch.extra, ch.rows = True, True, None, 0
                        chunks = [ch]
                    else:
                        chunks = self.rows_chunks(a0, a1, cr, H, True, True)
                else:
                    if a1 <= a0 and b1 <= b0:
                        ch = Chunk(); ch.first, ch.last, ch.extra, ch.rows = True, True, None, 0
                        chunks = [ch]
                    else:
                        if a1 > a0:
                            chunks += self.rows_chunks(a0, a1, cr, H, True, b1 <= b0, "rtr")
                        if b1 > b0:
                            chunks += self.rows_chunks(b0, b1, cr, H, a1 <= a0, True)
            for ch in chunks:
                if ch.first and l > 0:
                    ch.waits.append((("out", l - 1), self.target("out") + bump))
                if ch.extra == "rtr":
                    ch.arrives.append(("rtr", l))
                if ch.last and op == OP_P1:
                    ch.arrives.append(("p1", l))
            return chunks, None
        if op == OP_ROUTE:
            if self.one:
                return [Chunk()], (("rtr", l), self.target("rtr"))
            ch = Chunk(waits=[(("rtr", l), self.target("rtr"))])
            ch.routes = l
            return [ch], None
        if op == OP_ATTN:
            P, hkv, hd = d.page_size, d.n_kv_heads, d.head_dim
            pb = hkv * P * hd * 2
            pps = 1 if pb >= STAGE_BYTES // 2 else (STAGE_BYTES // 2) // pb
            it, off = self.plan["items"], self.plan["item_off"]
            for k in range(off[s], off[s + 1]):
                b, t0, t1 = int(it[k][0]), int(it[k][3]), int(it[k][4])
                npages = cdiv(t1, P) - t0 // P
                chunks.append(Chunk(waits=[(("p1", l), self.target("p1"))], stages=cdiv(npages, pps),
                                    arrives=[("items", l, b)]))
            return chunks, None
        if op == OP_COMBINE:
            meta = self.plan["meta"]
            waits = [(("items", l, u // d.n_q_heads), int(meta[u // d.n_q_heads][1])) for u in range(a0, a1)]
            return [Chunk(waits=waits, arrives=[("comb", l)])], None
        if op == OP_UP:
            n_act, cnt = self.active(l)
            if self.one:
                G = d.moe_inter // 8
                g0 = g1 = 0
                if a0 >= 0:
                    if a1 >= n_act:
                        a = ((a0 + 1) * n_act - 1) // a1
                        s0, s1 = a * a1 // n_act, (a + 1) * a1 // n_act
                        g0, g1 = dshare(G, s1 - s0, a0 - s0)
                        g0, g1 = g0 + a * G, g1 + a * G
                    else:
                        g0, g1 = dshare(n_act * G, a1, a0)
                self.coverage["up"].setdefault(l, []).append((g0, g1))
                g = g0
                while g < g1:
                    a = g // G
                    ge = min(g1, (a + 1) * G, g + 8)
                    ncb = ge - g
                    chunks.append(Chunk(stages=2 * cdiv(8 * ncb, rows_per_stage(H))
                                        + ncb * cdiv(H, rows_per_stage(8))))
                    g = ge
            else:
                p0 = p1 = 0
                if a0 >= 0:
                    p0, p1 = dshare(n_act * d.moe_inter, a1, a0)
                self.coverage["up"].setdefault(l, []).append((p0, p1))
                a = p0 // d.moe_inter
                while a < n_act and a * d.moe_inter < p1:
                    i0, i1 = max(p0 - a * d.moe_inter, 0), min(p1 - a * d.moe_inter, d.moe_inter)
                    cp = max(1, chunk_rows(H, cnt[a]) // 2)
                    c0 = i0
                    while c0 < i1:
                        chunks.append(Chunk(stages=2 * cdiv(min(cp, i1 - c0), rows_per_stage(H))))
                        c0 += cp
                    a += 1
            if not chunks:
                chunks = [Chunk()]
            chunks[-1].arrives.append(("up", l))
            return chunks, None
        if op == OP_OUT:
            KO = d.n_q_heads * d.head_dim
            if self.one or a1 <= a0:
                cr = one_rows(KO) if self.one else 1
                seq = []
                c0 = a0
                while c0 < a1:
                    seq.append(min(cr, a1 - c0))
                    c0 += cr
                if not seq:
                    seq = [0]
                for i, n in enumerate(seq):
                    ch = Chunk(stages=cdiv(n, rows_per_stage(KO)))
                    if n > 0:
                        ch.waits.append((("comb", l), self.target("comb")))
                    chunks.append(ch)
                chunks[-1].arrives.append(("out", l))
                return chunks, None
            co = chunk_rows(KO, B)
            c0 = a0
            while c0 < a1:
                n = min(co, a1 - c0)
                chunks.append(Chunk(waits=[(("comb", l), self.target("comb"))], stages=cdiv(n, rows_per_stage(KO))))
                c0 += co
            chunks.append(Chunk(waits=[(("down", l), self.target("down"))], arrives=[("out", l)]))
            return chunks, None
        if op == OP_DOWN:
            if self.one:
                self.coverage["down"].setdefault(l, []).append((a0, a1))
                ch = Chunk(arrives=[("out", l)])
                if a1 > a0:
                    ng = d.top_k * (d.moe_inter // 8)
                    nx = len(range(a0 & ~3, a1, 24))
                    ch.stages = nx * cdiv(ng, 256)
                    return [ch], ("after", (("up", l), self.target("up")))
                return [ch], None
            n_act, cnt = self.active(l)
            r0 = r1 = 0
            if a0 >= 0:
                r0, r1 = dshare(n_act * H, a1, a0)
            self.coverage["down"].setdefault(l, []).append((r0, r1))
            if r1 <= r0:
                return [Chunk(arrives=[("down", l)])], None
            a = r0 // H
            while a < n_act and a * H < r1:
                h0, h1 = max(r0 - a * H, 0), min(r1 - a * H, H)
                cd = chunk_rows(d.moe_inter, cnt[a])
                c0 = h0
                while c0 < h1:
                    n = min(cd, h1 - c0)
                    chunks.append(Chunk(waits=[(("up", l), self.target("up"))],
                                        stages=cdiv(n, rows_per_stage(d.moe_inter))))
                    c0 += cd
                a += 1
            chunks[-1].arrives.append(("down", l))
            return chunks, None
        raise ValueError(f"unknown op {op}")

    # ------------------------------------------------------ agents
    def claimed(self, s, t):
        """Several tokens, claimed tiles: the producer claims the next tile
        before it hands over the current one's chunks (so the last claimed
        tile's last chunk carries the arrival); an SM that claims nothing
        hands over one empty chunk that arrives."""
        d, H = self.d, self.d.hidden
        op, l, a0 = int(t[F_OP]), int(t[F_LAYER]), int(t[F_A0])
        n_act, cnt = self.active(l)
        up = op == OP_UP
        kind = "up" if up else "down"
        per, T = (d.moe_inter, max(1, self.claim_rows // 2)) if up else (H, self.claim_rows)
        tpe = cdiv(per, T)
        ntiles = n_act * tpe

        def claim():
            v = self.claims.get((kind, l), 0)
            self.claims[(kind, l)] = v + 1
            return v

        c = claim() if a0 >= 0 else ntiles
        if c >= ntiles:
            yield from self.hand_over(s, [Chunk(arrives=[(kind, l)])])
            return
        while c < ntiles:
            nx = claim()
            a, lo = c // tpe, (c % tpe) * T
            hi = min(lo + T, per)
            self.coverage[kind].setdefault(l, []).append((a * per + lo, a * per + hi))
            chunks = []
            step = max(1, chunk_rows(H, cnt[a]) // 2) if up else chunk_rows(d.moe_inter, cnt[a])
            c0 = lo
            while c0 < hi:
                n = min(step, hi - c0)
                if up:
                    chunks.append(Chunk(stages=2 * cdiv(n, rows_per_stage(H))))
                else:
                    chunks.append(Chunk(waits=[(("up", l), self.target("up"))],
                                        stages=cdiv(n, rows_per_stage(d.moe_inter))))
                c0 += step
            if nx >= ntiles:
                chunks[-1].arrives.append((kind, l))
            yield from self.hand_over(s, chunks)
            c = nx

    def hand_over(self, s, chunks):
        for ch in chunks:
            yield ("slot", s)
            self.handed[s] += 1
            self.queue[s].append(ch)
            for _ in range(ch.stages):
                yield ("stage", s)
                self.issued[s] += 1
                ch.issued += 1

    def producer(self, s):
        tasks = self.plan["tasks"][self.plan["task_off"][s]:self.plan["task_off"][s + 1]]
        for t in tasks:
            op, l = int(t[F_OP]), int(t[F_LAYER])
            if not self.one and op in (OP_UP, OP_DOWN):
                yield ("route", s, l)                   # the consumer has routed layer l
            if self.claim_rows and op in (OP_UP, OP_DOWN):
                yield from self.claimed(s, t)
                continue
            chunks, pw = self.resolve(s, t)
            if pw is not None and pw[0] != "after":
                yield ("ctr",) + pw                     # producer-side wait before the hand-over
            for ch in chunks:
                yield ("slot", s)
                self.handed[s] += 1
                self.queue[s].append(ch)
                if pw is not None and pw[0] == "after":
                    yield ("ctr",) + pw[1]
                for _ in range(ch.stages):
                    yield ("stage", s)
                    self.issued[s] += 1
                    ch.issued += 1
        yield ("slot", s)
        self.handed[s] += 1
        self.queue[s].append(Chunk(end=True))

    def consumer(self, s):
        while True:
            yield ("queue", s)
            ch = self.queue[s].pop(0)
            if ch.end:
                return
            for c, tgt in ch.waits:
                yield ("ctr", c, tgt)
            for k in range(ch.stages):
                yield ("arrived", ch, k)
                self.released[s] += 1
            if ch.routes >= 0:
                self.route_done[s] = ch.routes + 1
            for c in ch.arrives:
                self.counters[c] = self.counters.get(c, 0) + 1
            self.consumed[s] += 1

    def ready(self, cond):
        kind = cond[0]
        if kind == "ctr":
            return self.counters.get(cond[1], 0) >= cond[2]
        if kind == "slot":
            return self.handed[cond[1]] - self.consumed[cond[1]] < TASK_SLOTS
        if kind == "stage":
            return self.issued[cond[1]] - self.released[cond[1]] < STAGES
        if kind == "queue":
            return len(self.queue[cond[1]]) > 0
        if kind == "arrived":
            return cond[1].issued > cond[2]
        if kind == "route":
            return self.route_done[cond[1]] > cond[2]
        raise ValueError(kind)

    def run(self, seed=0, max_burst=8):
        rng = random.Random(seed)
        n = self.n_sm
        self.queue = [[] for _ in range(n)]
        self.handed, self.consumed = [0] * n, [0] * n
        self.issued, self.released = [0] * n, [0] * n
        agents = []
        for s in range(n):
            agents.append(["P", s, self.producer(s), None])
            agents.append(["C", s, self.consumer(s), None])
        for a in agents:
            a[3] = next(a[2])
        live = list(agents)
        while live:
            rng.shuffle(live)
            moved = False
            still = []
            for a in live:
                done = False
                for _ in range(rng.randint(1, max_burst)):
                    if not self.ready(a[3]):
                        break
                    moved = True
                    try:
                        a[3] = a[2].send(None)
                    except StopIteration:
                        done = True
                        break
                if not done:
                    still.append(a)
            live = still
            if live and not moved:
                stuck = []
                for a in live:
                    c = a[3]
                    if c[0] == "ctr":
                        stuck.append((a[0], a[1], c[1], self.counters.get(c[1], 0), c[2]))
                raise Deadlock(f"no agent can move; counter waits stuck (agent, SM, counter, value, "
                               f"target): {stuck[:8]}")
        return self.counters
