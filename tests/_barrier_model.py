"""A model of the mbarrier protocols of the warp-specialized branch-attention kernels
(csrc/attn.cu), run on the CPU under random schedules.  Test infrastructure only: it
checks the synchronisation design, not the arithmetic.

What is modelled:
* an mbarrier: an arrival count per phase, pending transaction bytes (expect_tx adds,
  the copy's completion removes) and a completed-phase counter; a parity wait for phase
  k returns once the counter's parity differs from k's, exactly as the hardware test
  does, so a wait that is two phases behind blocks and one whose barrier is a phase
  behind returns early;
* each issuing thread's tensor products and commits, executed in that thread's issue
  order (a commit arrives once everything the thread issued before it has executed),
  with the threads' queues drained in any interleaving and issue blocking while a
  queue is full;
* tiled copies that land at any later time;
* named barriers among a fixed group of warps;
* buffers with versions: a write stores (what, step), a read names the version it
  expects, so a product or a load that reads a slot already overwritten for a later
  step (or not yet written) is caught.

What is checked, under every schedule: no deadlock; every wait returns on exactly the
phase it waits for; no phase of a barrier that several warps arrive on completes with
arrivals of different steps; every read sees the version it expects.
"""
import random


class Violation(Exception):
    pass


class Barrier:
    def __init__(self, sim, name, count, tagged):
        self.sim, self.name, self.count, self.tagged = sim, name, count, tagged
        self.completed = 0
        self.arrived = 0
        self.tx = 0
        self.tags = []

    def arrive(self, tag):
        self.arrived += 1
        if self.arrived > self.count:
            self.sim.fail(f"{self.name}: more arrivals than its count")
        if self.tagged:
            self.tags.append(tag)
        self._maybe_complete()

    def complete_tx(self):
        self.tx -= 1
        self._maybe_complete()

    def _maybe_complete(self):
        if self.arrived == self.count and self.tx == 0:
            if self.tagged and len(set(self.tags)) > 1:
                self.sim.fail(f"{self.name}: phase {self.completed} mixes steps {sorted(set(self.tags))}")
            self.completed += 1
            self.arrived = 0
            self.tags = []


class Sim:
    """Agents are generators yielding actions:
      ('wait', bar, k)            wait for phase k of bar (parity wait)
      ('arrive', bar, tag)
      ('copy', bar, tag, buf, ver) expect_tx on bar (one arrival), a copy that later writes
                                  buf := ver and completes the transaction
      ('mma', issuer, reads, writes)  enqueue a product: reads = [(buf, ver)], writes =
                                  [(buf, ver)], executed later in the issuer's order
      ('commit', issuer, bar, tag)    enqueue a commit
      ('read', buf, ver)          a load by the agent itself (checked now)
      ('write', buf, ver)         a store by the agent itself
      ('sync', name, count)       named barrier among `count` agents
    """

    def __init__(self, seed, qmax=2):
        self.rng = random.Random(seed)
        self.qmax = qmax
        self.bars = {}
        self.bufs = {}
        self.queues = {}
        self.copies = []
        self.named = {}
        self.agents = []

    def fail(self, msg):
        raise Violation(msg)

    def bar(self, name, count=1, tagged=False):
        self.bars[name] = Barrier(self, name, count, tagged)
        return name

    def agent(self, gen):
        self.agents.append({"gen": gen, "act": None, "done": False})

    def _read(self, buf, ver, who):
        have = self.bufs.get(buf)
        if have != ver:
            self.fail(f"{who} read {buf} = {have}, expected {ver}")

    def _ready(self, a):
        act = a["act"]
        kind = act[0]
        if kind == "wait":
            b = self.bars[act[1]]
            return b.completed % 2 != act[2] % 2
        if kind in ("mma", "commit"):
            return len(self.queues.setdefault(act[1], [])) < self.qmax
        if kind == "sync":
            st = self.named.setdefault(act[1], {"waiting": 0, "gen": 0})
            return a.get("sync_gen") is not None and st["gen"] > a["sync_gen"]
        return True

    def _perform(self, a):
        act = a["act"]
        kind = act[0]
        if kind == "wait":
            b = self.bars[act[1]]
            if b.completed != act[2] + 1:
                self.fail(f"wait on {act[1]} for phase {act[2]} returned with {b.completed} phases complete")
        elif kind == "arrive":
            self.bars[act[1]].arrive(act[2])
        elif kind == "copy":
            b = self.bars[act[1]]
            b.tx += 1
            b.arrive(act[2])
            self.copies.append((act[1], act[3], act[4]))
        elif kind == "mma":
            self.queues.setdefault(act[1], []).append(("mma", act[2], act[3]))
        elif kind == "commit":
            self.queues.setdefault(act[1], []).append(("commit", act[2], act[3]))
        elif kind == "read":
            self._read(act[1], act[2], "agent")
        elif kind == "write":
            self.bufs[act[1]] = act[2]
        a["act"] = None
        a["sync_gen"] = None

    def _advance(self, a):
        try:
            a["act"] = next(a["gen"])
        except StopIteration:
            a["done"] = True
            return
        if a["act"][0] == "sync":
            st = self.named.setdefault(a["act"][1], {"waiting": 0, "gen": 0})
            a["sync_gen"] = st["gen"]
            st["waiting"] += 1
            if st["waiting"] == a["act"][2]:
                st["waiting"] = 0
                st["gen"] += 1

    def run(self, max_steps=200000):
        for a in self.agents:
            self._advance(a)
        for _ in range(max_steps):
            choices = []
            for a in self.agents:
                if not a["done"] and self._ready(a):
                    choices.append(("agent", a))
            for name, q in self.queues.items():
                if q:
                    choices.append(("pipe", name))
            for i in range(len(self.copies)):
                choices.append(("copy", i))
            if not choices:
                if all(a["done"] for a in self.agents):
                    return
                stuck = [a["act"] for a in self.agents if not a["done"]]
                self.fail(f"deadlock: {stuck[:4]}")
            kind, x = self.rng.choice(choices)
            if kind == "agent":
                if x["act"][0] != "sync":
                    self._perform(x)
                else:
                    x["act"] = None
                self._advance(x)
            elif kind == "pipe":
                op = self.queues[x].pop(0)
                if op[0] == "mma":
                    for buf, ver in op[1]:
                        self._read(buf, ver, f"product of {x}")
                    for buf, ver in op[2]:
                        self.bufs[buf] = ver
                else:
                    self.bars[op[1]].arrive(op[2])
            else:
                bar, buf, ver = self.copies.pop(x)
                self.bufs[buf] = ver
                self.bars[bar].complete_tx()
        self.fail("step limit")


# ---- the forward: two TMA loaders, an S issuer, an O issuer, softmax warps ----------------

def forward(sim, n_kt, warps=4, per_buffer_pf=True, shared_o_done=False):
    """S_j = Q K_j^T into S buffer j % 2; softmax reads S_j, writes P_j into P buffer j % 2;
    O += P_j V_j.  Three K slots, two V slots.  `per_buffer_pf=False` and
    `shared_o_done=True` restore an earlier design (one P-ready barrier for both buffers, and
    the final wait on a single O-done barrier), which the checker must reject."""
    W = warps
    bQ = sim.bar("Q")
    KF = [sim.bar(f"KF{i}") for i in range(3)]
    KE = [sim.bar(f"KE{i}") for i in range(3)]
    VF = [sim.bar(f"VF{i}") for i in range(2)]
    VE = [sim.bar(f"VE{i}") for i in range(2)]
    SF = [sim.bar(f"SF{i}") for i in range(2)]
    SE = [sim.bar(f"SE{i}", W, tagged=True) for i in range(2)]
    PF = [sim.bar(f"PF{i}", W, tagged=True) for i in range(2)] if per_buffer_pf else [sim.bar("PF", W, tagged=True)] * 2
    PD = [sim.bar(f"PD{i}") for i in range(2)]
    OD = sim.bar("OD")
    rng = sim.rng

    def k_loader():
        yield ("copy", bQ, 0, "Q", ("Q", 0))
        for kt in range(n_kt):
            s, use = kt % 3, kt // 3
            if use > 0:
                yield ("wait", KE[s], use - 1)
            yield ("copy", KF[s], kt, f"K{s}", ("K", kt))

    def v_loader():
        for kt in range(n_kt):
            s, use = kt % 2, kt // 2
            if use > 0:
                yield ("wait", VE[s], use - 1)
            yield ("copy", VF[s], kt, f"V{s}", ("V", kt))

    def s_issuer():
        yield ("wait", bQ, 0)
        for kt in range(n_kt):
            b, ks = kt & 1, kt % 3
            yield ("wait", KF[ks], kt // 3)
            if kt >= 2:
                yield ("wait", SE[b], (kt - 2) // 2)
            yield ("mma", "S", [("Q", ("Q", 0)), (f"K{ks}", ("K", kt))], [(f"S{b}", ("S", kt))])
            yield ("commit", "S", SF[b], kt)
            yield ("commit", "S", KE[ks], kt)

    def o_issuer():
        pf_phase = [0, 0]
        for kt in range(n_kt):
            b = kt & 1
            if per_buffer_pf:
                yield ("wait", PF[b], kt // 2)
            else:
                yield ("wait", PF[0], kt)
            yield ("wait", VF[b], kt // 2)
            yield ("mma", "O", [(f"P{b}r{r}", ("P", kt)) for r in range(W // 2)] + [(f"V{b}", ("V", kt))], [])
            yield ("commit", "O", PD[b], kt)
            yield ("commit", "O", VE[b], kt)
            if shared_o_done:
                yield ("commit", "O", OD, kt)

    def softmax(w):
        for kt in range(n_kt):
            b = kt & 1
            yield ("wait", SF[b], kt // 2)
            yield ("read", f"S{b}", ("S", kt))
            yield ("arrive", SE[b], kt)
            yield ("sync", f"row{w // 2}", 2)
            if kt >= 2:
                yield ("wait", PD[b], (kt - 2) // 2)
            yield ("write", f"P{b}r{w // 2}", ("P", kt))          # the row pair's rows of P
            if kt > 0 and rng.random() < 0.3:        # the running max moved: O is rescaled
                yield ("wait", PD[(kt - 1) & 1], (kt - 1) // 2)
            yield ("arrive", PF[b], kt)
        if shared_o_done:
            yield ("wait", OD, n_kt - 1)
        else:
            yield ("wait", PD[(n_kt - 1) & 1], (n_kt - 1) // 2)

    for g in (k_loader(), v_loader(), s_issuer(), o_issuer()):
        sim.agent(g)
    for w in range(W):
        sim.agent(softmax(w))


# ---- dQ: K loader (+ Q, dO), V loader, products issuer, dQ issuer, dS warps --------------

def dq(sim, n_kt, warps=4, wait_dp_read=True):
    """`wait_dp_read=False` drops the products thread's wait for every dS thread to have read
    dP_{j-1} before dP_j overwrites it (a planted mistake the checker must reject)."""
    W = warps
    bQ = sim.bar("Q")
    KF = [sim.bar(f"KF{i}") for i in range(3)]
    KE = [sim.bar(f"KE{i}") for i in range(3)]
    VF = [sim.bar(f"VF{i}") for i in range(2)]
    VE = [sim.bar(f"VE{i}") for i in range(2)]
    SP = [sim.bar(f"SP{i}") for i in range(2)]
    PE = sim.bar("PE", W, tagged=True)
    DS = [sim.bar(f"DS{i}", W, tagged=True) for i in range(2)]
    QD = [sim.bar(f"QD{i}") for i in range(2)]

    def k_loader():
        yield ("copy", bQ, 0, "Q", ("Q", 0))
        for j in range(n_kt):
            s, use = j % 3, j // 3
            if use > 0:
                yield ("wait", KE[s], use - 1)
            yield ("copy", KF[s], j, f"K{s}", ("K", j))

    def v_loader():
        for j in range(n_kt):
            s, use = j % 2, j // 2
            if use > 0:
                yield ("wait", VE[s], use - 1)
            yield ("copy", VF[s], j, f"V{s}", ("V", j))

    def products():
        yield ("wait", bQ, 0)
        for j in range(n_kt):
            b, ks = j & 1, j % 3
            yield ("wait", KF[ks], j // 3)
            if j >= 2:
                yield ("wait", QD[b], (j - 2) // 2)
            yield ("mma", "P", [("Q", ("Q", 0)), (f"K{ks}", ("K", j))], [(f"S{b}r{r}", ("S", j)) for r in range(2)])
            yield ("wait", VF[b], j // 2)
            if j >= 1 and wait_dp_read:
                yield ("wait", PE, j - 1)
            yield ("mma", "P", [("Q", ("Q", 0)), (f"V{b}", ("V", j))], [("dP", ("dP", j))])
            yield ("commit", "P", SP[b], j)
            yield ("commit", "P", VE[b], j)

    def dq_issuer():
        for j in range(n_kt):
            b = j & 1
            yield ("wait", DS[b], j // 2)
            yield ("mma", "D", [(f"S{b}r{r}", ("dS", j)) for r in range(2)] + [(f"K{j % 3}", ("K", j))], [])
            yield ("commit", "D", QD[b], j)
            yield ("commit", "D", KE[j % 3], j)

    def ds_warp(w):
        for j in range(n_kt):
            b = j & 1
            yield ("wait", SP[b], j // 2)
            yield ("read", f"S{b}r{w % 2}", ("S", j))
            yield ("read", "dP", ("dP", j))
            yield ("arrive", PE, j)
            yield ("sync", f"row{w % 2}", W // 2)
            yield ("write", f"S{b}r{w % 2}", ("dS", j))            # the row group's rows of dS
            yield ("arrive", DS[b], j)
        yield ("wait", QD[(n_kt - 1) & 1], (n_kt - 1) // 2)

    for g in (k_loader(), v_loader(), products(), dq_issuer()):
        sim.agent(g)
    for w in range(W):
        sim.agent(ds_warp(w))


# ---- dK / dV: loader, products issuer, update issuer, two work groups ---------------------

def dkdv(sim, n_e, warps_per_group=2, wait_release=True):
    """Each query tile e is two steps i = 2 e + g; step 2 e + 1 is empty for a tile of at most
    64 rows (no products; the barriers still advance).  `wait_release=False` drops the
    products thread's wait for the update two steps back (a planted mistake)."""
    W = warps_per_group
    empty = [sim.rng.random() < 0.3 for _ in range(n_e)]
    KV = sim.bar("KV")
    QF = [sim.bar(f"QF{i}", 2, tagged=True) for i in range(2)]
    QE = [sim.bar(f"QE{i}") for i in range(2)]
    SP = [sim.bar(f"SP{i}") for i in range(2)]
    DS = [sim.bar(f"DS{i}", W, tagged=True) for i in range(2)]
    DVK = [sim.bar(f"DVK{i}") for i in range(2)]
    n_st = 2 * n_e

    def loader():
        yield ("copy", KV, 0, "KV", ("KV", 0))
        for e in range(n_e):
            s, use = e & 1, e >> 1
            if use > 0:
                yield ("wait", QE[s], use - 1)
            yield ("copy", QF[s], e, f"Q{s}", ("Q", e))          # lane 0: expect_tx + copies
            yield ("write", f"L{s}", ("L", e))                  # lse, D, the decoded entry
            yield ("arrive", QF[s], e)                          # every lane after its writes

    def products():
        for i in range(n_st):
            e, b = i >> 1, i & 1
            if b == 0:
                if i == 0:
                    yield ("wait", KV, 0)
                yield ("wait", QF[e & 1], e >> 1)
                yield ("read", f"L{e & 1}", ("L", e))
            if i >= 2 and wait_release:
                yield ("wait", DVK[b], (i - 2) >> 1)
            if not (b == 1 and empty[e]):
                yield ("mma", "P", [("KV", ("KV", 0)), (f"Q{e & 1}", ("Q", e))], [(f"S{b}", ("S", i))])
            yield ("commit", "P", SP[b], i)

    def updates():
        for i in range(n_st):
            e, b = i >> 1, i & 1
            yield ("wait", DS[b], i >> 1)
            yield ("read", f"L{e & 1}", ("L", e))
            if not (b == 1 and empty[e]):
                yield ("mma", "U", [(f"S{b}", ("P", i)), (f"Q{e & 1}", ("Q", e))], [])
            yield ("commit", "U", DVK[b], i)
            if b == 1:
                yield ("commit", "U", QE[e & 1], e)

    def work(g, w):
        for e in range(n_e):
            i = 2 * e + g
            yield ("wait", QF[e & 1], e >> 1)
            yield ("read", f"L{e & 1}", ("L", e))
            yield ("wait", SP[g], e)
            if g == 1 and empty[e]:
                yield ("arrive", DS[g], i)
                continue
            yield ("read", f"S{g}", ("S", i))
            yield ("sync", f"g{g}", W)
            yield ("write", f"S{g}", ("P", i))
            yield ("arrive", DS[g], i)
        if g == 1 and n_e > 0:
            yield ("wait", DVK[1], n_e - 1)

    for gen in (loader(), products(), updates()):
        sim.agent(gen)
    for g in range(2):
        for w in range(W):
            sim.agent(work(g, w))
