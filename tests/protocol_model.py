"""A model of the two tensor-core kernels' synchronisation, for checking on the CPU.

compute-sanitizer (its race and barrier checks) cannot run here, so the mbarrier protocols of
the decode kernel (producer warps filling a ring of stages, consumer warps draining it) and of
the varlen kernel (producer, MMA issuer, one softmax group per query tile) are restated as Python
generators, role by role and wait by wait as the kernels do them, and run under random
interleavings. An mbarrier completes a phase when its arrivals for that phase are in; a
parity wait passes when the barrier's completed-phase count has the other parity. Copies land
in any order, tensor-core operations complete in issue order and a commit arrives when every
operation issued before it has completed. Checked on every run:
  - no deadlock;
  - every wait that passes waits for a phase that has completed, and none waits for a phase
    more than one behind (a parity wait cannot tell phase j from j - 2);
  - every product reads the ring tile it means to, and no buffer is overwritten while a reader
    still needs it (ring stages, score and output blocks); no output is read before its last
    product has landed;
  - when the roles are done (the CTA leaves), no copy or commit is still in flight.
This is a model of the protocol, not of the kernels' arithmetic: it has to change with them.
"""

from __future__ import annotations

import random


class ProtocolError(AssertionError):
    pass


class Barrier:
    def __init__(self, name: str, count: int):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: more arrivals than the phase expects")
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, phase: int) -> bool:
        ok = (self.done & 1) != (phase & 1)
        if ok and self.done <= phase:
            raise ProtocolError(f"{self.name}: wait for phase {phase} passed with {self.done} completed")
        if not ok and self.done > phase + 1:
            raise ProtocolError(f"{self.name}: wait for phase {phase} missed it ({self.done} completed)")
        return ok


class Machine:
    """Barriers, in-flight copies (land in any order) and the tensor pipe (in order)."""

    def __init__(self, seed: int):
        self.rng = random.Random(seed)
        self.bars: dict[str, Barrier] = {}
        self.copies: list[tuple[str, callable]] = []
        self.pipe: list[tuple[str, callable]] = []

    def bar(self, name: str, count: int = 1):
        self.bars[name] = Barrier(name, count)

    def copy(self, bar: str, on_land=None):
        self.copies.append((bar, on_land))

    def op(self, on_done=None):
        self.pipe.append(("op", on_done))

    def commit(self, bar: str):
        self.pipe.append(("commit", bar))

    def run(self, roles: dict):
        waiting = {k: None for k in roles}
        alive = set(roles)
        for _ in range(10 ** 6):
            if not alive and not self.copies and not self.pipe:
                return
            ready = [("role", k) for k in sorted(alive)
                     if waiting[k] is None or waiting[k][0] == "step" or
                     self.bars[waiting[k][1]].passes(waiting[k][2])]
            if self.copies:
                ready.append(("copy", None))
            if self.pipe:
                ready.append(("pipe", None))
            if not ready:
                raise ProtocolError(f"deadlock: {[(k, waiting[k]) for k in sorted(alive)]}")
            kind, k = self.rng.choice(ready)
            if kind == "copy":
                bar, on_land = self.copies.pop(self.rng.randrange(len(self.copies)))
                if on_land:
                    on_land()
                self.bars[bar].arrive()
            elif kind == "pipe":
                what, x = self.pipe.pop(0)
                if what == "commit":
                    self.bars[x].arrive()
                elif x:
                    x()
            else:
                try:
                    waiting[k] = next(roles[k])
                except StopIteration:
                    alive.discard(k)
                    waiting[k] = None
                    if not alive and (self.copies or any(w == "commit" for w, _ in self.pipe)):
                        raise ProtocolError("the CTA leaves with copies or commits in flight")
        raise ProtocolError("no progress")


def wait(bar: str, phase: int):
    return ("wait", bar, phase)


STEP = ("step",)


# ------------------------------------------------------------------ decode ring
def decode_ring(chunks: int, stages: int, producers: int, consumers: int, seed: int,
                release_early: bool = True):
    """Producer warp w copies chunks w, w + producers, ... into stage i % stages once the stage's
    previous chunk is released; consumer warp c takes chunks c, c + consumers, ...; 8-bit caches
    release a stage as soon as its codes are in registers (release_early), bf16 after P.V."""
    m = Machine(seed)
    for s in range(stages):
        m.bar(f"full{s}")
        m.bar(f"empty{s}")
    holder = {}  # stage -> chunk whose data is in it and still needed

    def producer(w):
        for i in range(w, chunks, producers):
            st = i % stages
            if i >= stages:
                yield wait(f"empty{st}", i // stages - 1)
            if st in holder:
                raise ProtocolError(f"stage {st} refilled (chunk {i}) while chunk {holder[st]} still needs it")
            holder[st] = i
            m.copy(f"full{st}")

    def consumer(c):
        for i in range(c, chunks, consumers):
            st = i % stages
            yield wait(f"full{st}", i // stages)
            if holder.get(st) != i:
                raise ProtocolError(f"chunk {i} read stage {st} holding {holder.get(st)}")
            if not release_early:
                yield STEP  # the products still read the stage
            del holder[st]
            m.bars[f"empty{st}"].arrive()
            yield STEP

    roles = {f"p{w}": producer(w) for w in range(producers)}
    roles.update({f"c{c}": consumer(c) for c in range(consumers)})
    m.run(roles)


# ------------------------------------------------------------------ varlen tile pair
def varlen_pair(nA: int, nB: int, seed: int, stages: int = 2, conditional_release: bool = True,
                score_phase_offset: int = 0):
    """One CTA: query tiles A and B (nA, nB key tiles; nB is 0 or >= nA), a `stages`-deep K and V
    ring, S_t and O_t blocks in TMEM, the MMA issue order S_A(0), S_B(0), then per key tile
    P.V_A(j), S_A(j+1), P.V_B(j), S_B(j+1); a ring stage released only if a later tile refills it
    (conditional_release)."""
    m = Machine(seed)
    n = max(nA, nB)
    for name in ["Q"] + [f"{x}{s}" for x in ("KF", "VF", "KE", "VE") for s in range(stages)] + \
            [f"{x}{t}" for x in ("SF", "PR", "OD") for t in range(2)]:
        m.bar(name)
    state = {"stage_readers": {}, "content": {}, "softmax_in": [False, False], "pv_left": [0, 0]}
    ntile = (nA, nB)

    def producer():
        m.copy("Q")
        for i in range(n):
            st = i % stages
            for x, rel in (("K", "KE"), ("V", "VE")):
                if i >= stages:
                    yield wait(f"{rel}{st}", i // stages - 1)
                if state["stage_readers"].get((x, st), 0):
                    raise ProtocolError(f"{x} stage {st} refilled while the tensor pipe reads it")
                state["content"][(x, st)] = i
                m.copy(f"{x}F{st}")

    def issue(kind, t, tile):
        key = ("K" if kind == "S" else "V", tile % stages)
        if state["content"].get(key) != tile:
            raise ProtocolError(f"{kind}_{t} of tile {tile} issued on stage holding {state['content'].get(key)}")
        state["stage_readers"][key] = state["stage_readers"].get(key, 0) + 1
        if kind == "PV":
            state["pv_left"][t] += 1

        def done():
            if state["content"].get(key) != tile:
                raise ProtocolError(f"{kind}_{t} of tile {tile} read a refilled stage")
            state["stage_readers"][key] -= 1
            if kind == "S":
                if state["softmax_in"][t]:
                    raise ProtocolError(f"S_{t} overwritten while its softmax reads it")
            else:
                state["pv_left"][t] -= 1
        m.op(done)
        m.commit(("SF" if kind == "S" else "OD") + str(t))

    def release(cond, bar):
        if cond or not conditional_release:
            m.commit(bar)

    def mma():
        yield wait("Q", 0)
        yield wait("KF0", 0)
        if nA:
            issue("S", 0, 0)
        if nB:
            issue("S", 1, 0)
        release(stages < n, "KE0")
        for j in range(n):
            st = j % stages
            yield wait(f"VF{st}", j // stages)
            if j < nA:
                yield wait("PR0", j)
                issue("PV", 0, j)
            nxt = j + 1 < n
            if nxt:
                yield wait(f"KF{(j + 1) % stages}", (j + 1) // stages)
                if j + 1 < nA:
                    issue("S", 0, j + 1)
            if j < nB:
                yield wait("PR1", j)
                issue("PV", 1, j)
            release(j + stages < n, f"VE{st}")
            if nxt:
                if j + 1 < nB:
                    issue("S", 1, j + 1)
                release(j + 1 + stages < n, f"KE{(j + 1) % stages}")

    def softmax(t):
        k = ntile[t]
        for j in range(k):
            yield wait(f"SF{t}", j + score_phase_offset)
            state["softmax_in"][t] = True
            yield STEP
            state["softmax_in"][t] = False
            m.bars[f"PR{t}"].arrive()
        if k:
            yield wait(f"OD{t}", k - 1)
            if state["pv_left"][t]:
                raise ProtocolError(f"O_{t} read before its last P.V landed")

    m.run({"producer": producer(), "mma": mma(), "softmaxA": softmax(0), "softmaxB": softmax(1)})


# ------------------------------------------------------------------ varlen lone tile
def varlen_lone(nA: int, seed: int, stages: int = 3, merge_wait: bool = True, lead: int = 1):
    """One CTA whose second query tile is empty: a `stages`-deep K and V ring; the two softmax
    groups take the key tiles in turn (tile j: group j % 2, score block j % 2, O block j % 2); the
    MMA issue order S(0), S(1), then per key tile P.V(j), S(j+2). At the end group 1 hands its
    row state to group 0 through K stage 0 (a named barrier) and group 0 merges O block 1 into
    its own (merge_wait: group 0 waits at the named barrier first). The producer's K copies run
    `lead` tiles ahead of its V copies."""
    m = Machine(seed)
    for name in ["Q", "NB"] + [f"{x}{s}" for x in ("KF", "VF", "KE", "VE") for s in range(stages)] + \
            [f"{x}{b}" for x in ("SF", "PR", "OD") for b in range(2)]:
        m.bar(name)
    state = {"stage_readers": {}, "content": {}, "softmax_in": [False, False], "p_readers": [0, 0],
             "pv_left": [0, 0], "handed": False}

    def producer():
        m.copy("Q")
        for e in range(nA + lead):
            for x, rel, i in (("K", "KE", e), ("V", "VE", e - lead)):
                if not 0 <= i < nA:
                    continue
                st = i % stages
                if i >= stages:
                    yield wait(f"{rel}{st}", i // stages - 1)
                if state["stage_readers"].get((x, st), 0):
                    raise ProtocolError(f"{x} stage {st} refilled while the tensor pipe reads it")
                if x == "K" and st == 0 and state["handed"]:
                    raise ProtocolError("K stage 0 refilled after the hand-over wrote it")
                state["content"][(x, st)] = i
                m.copy(f"{x}F{st}")

    def issue(kind, tile):
        key, b = ("K" if kind == "S" else "V", tile % stages), tile & 1
        if state["content"].get(key) != tile:
            raise ProtocolError(f"{kind} of tile {tile} issued on stage holding {state['content'].get(key)}")
        state["stage_readers"][key] = state["stage_readers"].get(key, 0) + 1
        if kind == "PV":
            state["pv_left"][b] += 1
            state["p_readers"][b] += 1

        def done():
            if state["content"].get(key) != tile:
                raise ProtocolError(f"{kind} of tile {tile} read a refilled stage")
            if key == ("K", 0) and state["handed"]:
                raise ProtocolError("S read K stage 0 after the hand-over wrote it")
            state["stage_readers"][key] -= 1
            if kind == "S":
                if state["softmax_in"][b] or state["p_readers"][b]:
                    raise ProtocolError(f"score block {b} overwritten while it is still read")
            else:
                state["pv_left"][b] -= 1
                state["p_readers"][b] -= 1
        m.op(done)
        m.commit(f"SF{b}" if kind == "S" else f"OD{b}")
        if kind == "S" and tile + stages < nA:
            m.commit(f"KE{tile % stages}")

    def mma():
        yield wait("Q", 0)
        for j in range(min(2, nA)):
            yield wait(f"KF{j}", 0)
            issue("S", j)
        for j in range(nA):
            st = j % stages
            yield wait(f"VF{st}", j // stages)
            yield wait(f"PR{j & 1}", j >> 1)
            issue("PV", j)
            if j + stages < nA:
                m.commit(f"VE{st}")
            if j + 2 < nA:
                yield wait(f"KF{(j + 2) % stages}", (j + 2) // stages)
                issue("S", j + 2)

    def softmax(t):
        n_mine = (nA + 1 - t) // 2
        for k in range(n_mine):
            yield wait(f"SF{t}", k)
            state["softmax_in"][t] = True
            yield STEP
            if k > 0 and state["pv_left"][t]:  # O_t rescaled (in the worst case, every tile)
                raise ProtocolError(f"O_{t} rescaled while a P.V still accumulates into it")
            state["softmax_in"][t] = False
            m.bars[f"PR{t}"].arrive()
        if n_mine:
            yield wait(f"OD{t}", n_mine - 1)
            if state["pv_left"][t]:
                raise ProtocolError(f"O_{t} read before its last P.V landed")
        if nA > 1:
            if t == 1:
                if state["stage_readers"].get(("K", 0), 0) or any(b == "KF0" for b, _ in m.copies):
                    raise ProtocolError("the hand-over wrote K stage 0 while it is still in use")
                state["handed"] = True
                m.bars["NB"].arrive()
            else:
                if merge_wait:
                    yield wait("NB", 0)
                if not state["handed"] or state["pv_left"][1]:
                    raise ProtocolError("group 0 merged before group 1's state and O block were final")

    m.run({"producer": producer(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)})
