"""Host-side model of the tensor-core forward kernel's barrier protocol.

Each role of a CTA (Q, K, V and rab producers, the score-product and PV issuers or the
single serial issuer, and every epilogue warp on its own) is a generator that issues the
same sequence of mbarrier waits and arrivals as the kernel, with the kernel's ring-slot
and parity formulas (slot = n % depth, wait parity = (n / depth) & 1, producer-side waits
on the phase before). TMA loads complete asynchronously in any order; tcgen05 products
and their commits run on one in-order tensor queue. A random scheduler interleaves the
roles and the completions.

Checks, at every step of every schedule:
  * a parity wait that passes must pass on exactly the phase it means (the barrier's
    completed-phase count is n + 1 for phase n): a count of n - 1 (a stale phase with
    the same parity) or n + 3 (an overrun) is a violation;
  * every buffer read (an S, P, K, V, Q or rab slot) finds the tile it expects;
  * the run ends with every role finished (no wait that never completes).
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field


class Violation(AssertionError):
    pass


class Barrier:
    def __init__(self, name: str, count: int):
        self.name, self.count = name, count
        self.pending = 0
        self.done = 0  # completed phases

    def arrive(self, n: int = 1):
        self.pending += n
        if self.pending > self.count:
            raise Violation(f"{self.name}: {self.pending} arrivals for a count of {self.count}")
        if self.pending == self.count:
            self.pending = 0
            self.done += 1


@dataclass
class Cfg:
    """Ring depths and roles of one kernel variant (the kernel's Cfg for a head dim)."""
    D: int
    NQ: int
    NK: int
    NV: int
    NR: int           # rab ring depth (0: no rab)
    NSB: int          # S buffers
    NPB: int          # P buffers (P over S: equal to NSB)
    NO: int           # O accumulators
    EPI_GROUPS: int   # epilogue groups taking alternate tiles
    SERIAL: bool      # one issuer, P written over S (S(t + NSB) waits for PV(t))
    warps_per_group: int = 2
    info_depth: int = 8
    # the D = 256 rab-ring guard (a group first waits for the other group's release of
    # tile t - 1 when the rab ring is shallower than the number of groups)
    rab_guard: bool = True
    # rab added by the tensor core: the score issuer consumes the rab ring (its product
    # accumulates the rab tile into S) and releases each slot with a commit
    RM: bool = False
    # K chunks per tile (head dim 512: eight 64-column chunks, each its own ring slot) and
    # V slots per tile (head dim 512: two 64-key halves)
    KCH: int = 1
    VCH: int = 1


# The kernel's configurations (four warps per group are modelled as fewer: the barrier
# counts scale with them, the protocol does not depend on the number).
def kernel_cfg(D: int, rab: bool, rab_mode: str = "epi") -> Cfg:
    """rab_mode: "epi" (rab or a custom mask read by the epilogue), "mma" (rab added by the
    tensor core, D <= 64), "two" (rab and a custom mask in one slot, D <= 128). D = 512:
    Q resident, K in 64-column chunks through a two-slot ring, one V tile, P over S."""
    if D == 512:
        return Cfg(D=D, NQ=1, NK=4, NV=1, NR=0, NSB=2, NPB=2, NO=1, EPI_GROUPS=2,
                   SERIAL=True, KCH=8, VCH=2)
    NQ = 2 if (D <= 64 or (D == 128 and not rab)) else 1
    NK = {32: 4, 64: 3 if rab else 4, 128: 2, 256: 1}[D]
    NV = 2 if (D == 64 and rab) else NK
    if not rab:
        NR = 0
    elif rab_mode == "two":
        NR = 2 if D == 32 else 1
    else:
        NR = {32: 4, 64: 3, 128: 2, 256: 1}[D]
    serial = D == 256
    # two O accumulators where TMEM has room beside two S buffers and two P buffers
    return Cfg(D=D, NQ=NQ, NK=NK, NV=NV, NR=NR, NSB=2, NPB=2, NO=2 if D <= 64 else 1,
               EPI_GROUPS=2 if serial else 1, SERIAL=serial, RM=rab and rab_mode == "mma")


@dataclass
class World:
    cfg: Cfg
    items: list               # n_kv of each work item, in claim order
    rng: random.Random
    bars: dict = field(default_factory=dict)
    slots: dict = field(default_factory=dict)   # (buffer, slot) -> tag of its contents
    tma: list = field(default_factory=list)     # pending async loads: (bar, buffer, slot, tag)
    tensor: list = field(default_factory=list)  # in-order queue of products / commits

    def bar(self, name, i=0):
        return self.bars[(name, i)]

    def check(self, buf, slot, want):
        got = self.slots.get((buf, slot))
        if got != want:
            raise Violation(f"{buf}[{slot}] holds {got}, reader expects {want}")

    # S and P buffers live in TMEM: every epilogue warp of the group that owns a buffer
    # reads and writes its own lanes / columns of it (a region per warp), while a product
    # writes (S) or reads (P) the regions of all of them.
    def regions(self, slot):
        c = self.cfg
        g = slot % c.EPI_GROUPS
        return [g * c.warps_per_group + i for i in range(c.warps_per_group)]

    def tensor_read(self, buf, slot, want):
        if buf in ("S", "P"):
            for r in self.regions(slot):
                self.check(buf, (slot, r), want)
        else:
            self.check(buf, slot, want)

    def tensor_write(self, buf, slot, tag):
        if buf in ("S", "P"):
            for r in self.regions(slot):
                self.slots[(buf, (slot, r))] = tag
        else:
            self.slots[(buf, slot)] = tag


def make_world(cfg: Cfg, items, seed: int) -> World:
    w = World(cfg=cfg, items=list(items), rng=random.Random(seed))
    gw = cfg.warps_per_group
    epi_warps = gw * cfg.EPI_GROUPS
    readers = epi_warps + (3 if cfg.SERIAL else 4) + (1 if cfg.NR else 0)

    def add(name, n, count):
        for i in range(n):
            w.bars[(name, i)] = Barrier(f"{name}[{i}]", count)
    add("q_full", cfg.NQ, 1)
    add("q_empty", cfg.NQ, 1)
    add("k_full", cfg.NK, 1)
    add("k_empty", cfg.NK, 1)
    add("v_full", cfg.NV, 1)
    add("v_empty", cfg.NV, 1)
    add("r_full", max(cfg.NR, 1), 1)
    add("r_empty", max(cfg.NR, 1), 1 if cfg.RM else gw)
    add("s_full", cfg.NSB, 1)
    add("s_free", cfg.NSB, gw)
    add("p_full", cfg.NPB, gw)
    add("pv_done", cfg.NPB, 1)
    add("o_full", cfg.NO, 1)
    add("o_empty", cfg.NO, epi_warps)
    add("info_full", cfg.info_depth, 1)
    add("info_empty", cfg.info_depth, readers)
    return w


# ----------------------------------------------------------------- actions
# A role yields ("wait", bar, n) to wait for the completion of phase n of bar (the kernel's
# parity wait with parity n & 1), ("arrive", bar), ("load", bar, buf, slot, tag) for a TMA
# load that arrives on bar when it lands, ("mma", [(buf, slot, tag) reads], (buf, slot, tag)
# write) and ("commit", bar) for the tensor queue, ("read", buf, slot, tag) and
# ("write", buf, slot, tag) for the epilogue's own accesses.
def _prod_wait(bar, it, depth):
    """A producer's wait for slot it % depth to be free (the phase before, skipped on the
    ring's first pass: the kernel's parity ((it / depth) & 1) ^ 1 passes at once there)."""
    return [] if it < depth else [("wait", bar, it // depth - 1)]


def q_producer(w: World):
    c = w.cfg
    q_it = 0
    for k, n in enumerate(w.items + [-1]):
        s = k % c.info_depth
        if k >= c.info_depth:
            yield ("wait", ("info_empty", s), k // c.info_depth - 1)
        w.slots[("info", s)] = k
        yield ("arrive", ("info_full", s))
        if n < 0:
            return
        qs = q_it % c.NQ
        for a in _prod_wait(("q_empty", qs), q_it, c.NQ):
            yield a
        yield ("load", ("q_full", qs), "Q", qs, k)
        q_it += 1


def _get_item(w, k):
    s = k % w.cfg.info_depth
    yield ("wait", ("info_full", s), k // w.cfg.info_depth)
    yield ("read", "info", s, k)
    yield ("arrive", ("info_empty", s))


def kv_producer(w: World, name):  # "K" or "V"
    c = w.cfg
    depth = c.NK if name == "K" else c.NV
    full, empty = ("k_full", "k_empty") if name == "K" else ("v_full", "v_empty")
    it = 0
    tile = 0
    for k, n in enumerate(w.items + [-1]):
        yield from _get_item(w, k)
        if n < 0:
            return
        for j in range(n):
            chunks = c.KCH if name == "K" else c.VCH
            for ch in range(chunks):
                s = it % depth
                for a in _prod_wait((empty, s), it, depth):
                    yield a
                yield ("load", (full, s), name, s, (tile, ch) if chunks > 1 else tile)
                it += 1
            tile += 1


def rab_producer(w: World):
    c = w.cfg
    it = 0
    for k, n in enumerate(w.items + [-1]):
        yield from _get_item(w, k)
        if n < 0:
            return
        for j in range(n):
            s = it % c.NR
            for a in _prod_wait(("r_empty", s), it, c.NR):
                yield a
            yield ("load", ("r_full", s), "R", s, it)
            it += 1


def s_issuer(w: World):
    """Score products S(t) = Q K(t)^T into S buffer t % NSB (own P buffers)."""
    c = w.cfg
    q_it = t = k_it = 0
    for k, n in enumerate(w.items + [-1]):
        yield from _get_item(w, k)
        if n < 0:
            return
        qs = q_it % c.NQ
        yield ("wait", ("q_full", qs), q_it // c.NQ)
        for j in range(n):
            sb, ks = t % c.NSB, k_it % c.NK
            if t >= c.NSB:
                yield ("wait", ("s_free", sb), t // c.NSB - 1)
            yield ("wait", ("k_full", ks), k_it // c.NK)
            yield ("mma", [("Q", qs, k), ("K", ks, t)], ("S", sb, ("S", t)))
            if c.RM:  # S += R (c I16): the rab tile of t, released by the commit
                rs = t % c.NR
                yield ("wait", ("r_full", rs), t // c.NR)
                yield ("mma", [("R", rs, t), ("S", sb, ("S", t))], ("S", sb, ("S", t)))
                yield ("commit", ("r_empty", rs))
            yield ("commit", ("s_full", sb))
            yield ("commit", ("k_empty", ks))
            if j + 1 == n:
                yield ("commit", ("q_empty", qs))
            k_it += 1
            t += 1
        q_it += 1


def pv_issuer(w: World):
    c = w.cfg
    t = v_it = u = 0
    for k, n in enumerate(w.items + [-1]):
        yield from _get_item(w, k)
        if n < 0:
            return
        ob = u % c.NO
        for j in range(n):
            pb, vs = t % c.NPB, v_it % c.NV
            yield ("wait", ("p_full", pb), t // c.NPB)
            yield ("wait", ("v_full", vs), v_it // c.NV)
            if j == 0 and u >= c.NO:
                yield ("wait", ("o_empty", ob), u // c.NO - 1)
            yield ("mma", [("P", pb, t), ("V", vs, t)], ("O", ob, k))
            yield ("commit", ("v_empty", vs))
            yield ("commit", ("pv_done", pb))
            v_it += 1
            t += 1
        yield ("commit", ("o_full", ob))
        u += 1


def serial_issuer(w: World):
    """One issuer, P over S: S(t0), S(t0 + 1), then per tile PV(t), S(t + 2)."""
    c = w.cfg
    q_it = k_it = v_it = u = 0
    t_base = 0

    def issue_s(t, qs, item):
        nonlocal k_it
        sb = t % c.NSB
        if t >= c.NSB:
            yield ("wait", ("pv_done", sb), t // c.NSB - 1)
        if c.KCH > 1:  # one product and one slot release per K chunk
            for ch in range(c.KCH):
                ks = k_it % c.NK
                yield ("wait", ("k_full", ks), k_it // c.NK)
                yield ("mma", [("Q", qs, item), ("K", ks, (t, ch))], ("S", sb, ("S", t)))
                yield ("commit", ("k_empty", ks))
                k_it += 1
            yield ("commit", ("s_full", sb))
            return
        ks = k_it % c.NK
        yield ("wait", ("k_full", ks), k_it // c.NK)
        yield ("mma", [("Q", qs, item), ("K", ks, t)], ("S", sb, ("S", t)))
        yield ("commit", ("s_full", sb))
        yield ("commit", ("k_empty", ks))
        k_it += 1

    def issue_pv(t, first, item):
        nonlocal v_it
        sb = t % c.NSB
        if first and u >= 1:
            yield ("wait", ("o_empty", 0), u - 1)
        for ch in range(c.VCH):  # one V slot per chunk of keys
            vs = v_it % c.NV
            yield ("wait", ("v_full", vs), v_it // c.NV)
            yield ("mma", [("S", sb, ("P", t)), ("V", vs, (t, ch) if c.VCH > 1 else t)],
                   ("O", 0, item))
            yield ("commit", ("v_empty", vs))
            v_it += 1
        yield ("commit", ("pv_done", sb))

    for k, n in enumerate(w.items + [-1]):
        yield from _get_item(w, k)
        if n < 0:
            return
        qs = q_it % c.NQ
        yield ("wait", ("q_full", qs), q_it // c.NQ)
        yield from issue_s(t_base, qs, k)
        if n >= 2:
            yield from issue_s(t_base + 1, qs, k)
        if n <= 2:
            yield ("commit", ("q_empty", qs))
        for j in range(n):
            t = t_base + j
            yield ("wait", ("p_full", t % c.NSB), t // c.NSB)
            yield from issue_pv(t, j == 0, k)
            if j + 2 < n:
                yield from issue_s(t + 2, qs, k)
                if j + 3 == n:
                    yield ("commit", ("q_empty", qs))
        t_base += n
        yield ("commit", ("o_full", 0))
        q_it += 1
        u += 1


def epilogue_warp(w: World, group: int, wid: int):
    """One epilogue warp (id wid) of `group` (tiles t with t % EPI_GROUPS == group)."""
    c = w.cfg
    t = u = 0
    prev = None  # item whose O is still to be drained
    rab = c.NR > 0 and not c.RM  # (RM: the score issuer reads rab)

    def drain(item):
        nonlocal u
        ob = u % c.NO
        yield ("wait", ("o_full", ob), u // c.NO)
        yield ("read", "O", ob, item)
        yield ("arrive", ("o_empty", ob))
        s = item % c.info_depth
        yield ("read", "info", s, item)
        yield ("arrive", ("info_empty", s))
        u += 1

    for k, n in enumerate(w.items + [-1]):
        s = k % c.info_depth
        yield ("wait", ("info_full", s), k // c.info_depth)
        yield ("read", "info", s, k)
        if n < 0:
            break
        gtile = 0
        for j in range(n):
            if t % c.EPI_GROUPS != group:
                t += 1
                continue
            sb = t % c.NSB
            yield ("wait", ("s_full", sb), t // c.NSB)
            if rab:
                rs = t % c.NR
                if c.rab_guard and c.NR < c.EPI_GROUPS and t >= 1:
                    yield ("wait", ("r_empty", (t - 1) % c.NR), (t - 1) // c.NR)
                yield ("wait", ("r_full", rs), t // c.NR)
                yield ("read", "R", rs, t)
            yield ("read", "S", (sb, wid), ("S", t))
            if not c.SERIAL:
                yield ("arrive", ("s_free", sb))
                pb = t % c.NPB
                if t >= c.NPB:
                    yield ("wait", ("pv_done", pb), t // c.NPB - 1)
                yield ("write", "P", (pb, wid), t)
            else:
                yield ("write", "S", (sb, wid), ("P", t))  # P over the S columns it read
            if rab:
                yield ("arrive", ("r_empty", rs))
            yield ("arrive", ("p_full", t % c.NPB))
            gtile += 1
            if prev is not None and (gtile == 1 or j + c.EPI_GROUPS >= n):
                yield from drain(prev)
                prev = None
            t += 1
        if prev is not None:
            yield from drain(prev)
        prev = k
    if prev is not None:
        yield from drain(prev)


# ----------------------------------------------------------------- scheduler
def run(cfg: Cfg, items, seed: int, max_steps: int = 10 ** 6, p_async: float = 0.5):
    """One random schedule; raises Violation on a broken invariant or a hang. p_async is
    the chance that a step completes an asynchronous operation (a TMA load or the head of
    the tensor queue) rather than advancing a role, when both are possible: low values
    let roles run far ahead of slow loads and products."""
    w = make_world(cfg, items, seed)
    roles = {"Q": q_producer(w), "K": kv_producer(w, "K"), "V": kv_producer(w, "V")}
    if cfg.NR:
        roles["R"] = rab_producer(w)
    if cfg.SERIAL:
        roles["MMA"] = serial_issuer(w)
    else:
        roles["S"] = s_issuer(w)
        roles["PV"] = pv_issuer(w)
    for g in range(cfg.EPI_GROUPS):
        for i in range(cfg.warps_per_group):
            roles[f"E{g}.{i}"] = epilogue_warp(w, g, g * cfg.warps_per_group + i)
    cur = {r: next(g) for r, g in roles.items()}
    done = set()

    def ready(a):
        if a[0] != "wait":
            return True
        b = w.bars[a[1]]
        return (b.done & 1) != (a[2] & 1)  # parity of phase n has completed

    for _ in range(max_steps):
        choices = [r for r in cur if r not in done and ready(cur[r])]
        n_async = len(w.tma) + (1 if w.tensor else 0)
        if not choices and n_async == 0:
            if len(done) == len(roles):
                return w
            stuck = {r: cur[r] for r in cur if r not in done}
            raise Violation(f"hang: {stuck}")
        if choices and (n_async == 0 or w.rng.random() >= p_async):
            pick = w.rng.randrange(len(choices))
        else:
            pick = len(choices) + w.rng.randrange(n_async)
        if pick >= len(choices):  # an asynchronous completion
            j = pick - len(choices)
            if j < len(w.tma):
                bar, buf, slot, tag = w.tma.pop(j)
                w.slots[(buf, slot)] = tag
                w.bars[bar].arrive()
            else:
                op = w.tensor.pop(0)
                if op[0] == "mma":
                    for buf, slot, tag in op[1]:
                        w.tensor_read(buf, slot, tag)
                    w.tensor_write(*op[2])  # an O accumulator holds its item
                else:
                    w.bars[op[1]].arrive()
            continue
        r = choices[pick]
        a = cur[r]
        if a[0] == "wait":
            b = w.bars[a[1]]
            if b.done != a[2] + 1:
                raise Violation(f"{r}: wait for phase {a[2]} of {b.name} passed with "
                                f"{b.done} phases completed")
        elif a[0] == "arrive":
            w.bars[a[1]].arrive()
        elif a[0] == "load":
            w.tma.append((a[1], a[2], a[3], a[4]))
        elif a[0] in ("mma", "commit"):
            w.tensor.append(a)
        elif a[0] == "read":
            w.check(a[1], a[2], a[3])
        elif a[0] == "write":
            w.slots[(a[1], a[2])] = a[3]
        try:
            cur[r] = next(roles[r])
        except StopIteration:
            done.add(r)
    raise Violation("schedule did not finish")
