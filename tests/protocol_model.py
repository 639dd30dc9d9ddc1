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
