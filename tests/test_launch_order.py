"""Host model of the ordering between kernels launched as programmatic dependents (CUDA's
programmatic stream serialization), as the library uses it: the backward's preprocess, dK/dV
and dQ kernels, and the decode's split and combine kernels, between other work on the stream.

Semantics modelled, for kernels K_1, K_2, ... queued in that order on one stream:
  - a kernel launched without the attribute begins once its predecessor has completed;
  - a kernel launched with it begins once its predecessor has triggered: every CTA of the
    predecessor has run `griddepcontrol.launch_dependents`, or the predecessor has completed
    (a kernel that never runs the instruction triggers at its completion);
  - `griddepcontrol.wait` in a kernel returns once its predecessor has completed (and that
    kernel's writes are visible);
  - a kernel completes after every step of its own.
The steps of each kernel are in program order.  From these rules the model builds the
happens-before relation over all steps and checks that every pair of accesses to one buffer by
two kernels, at least one a write, is ordered as the stream order says it must be.  The
kernels' step lists follow the launch code and the kernels' entry sequences (set-up, wait,
trigger, reads, writes); mutations drop one wait or trigger and must be caught."""
import itertools

import pytest


class Kernel:
    def __init__(self, name, steps, pdl):
        """steps: a list of ("wait",), ("trigger",), ("read", buf...), ("write", buf...)."""
        self.name, self.steps, self.pdl = name, steps, pdl


def happens_before(kernels):
    """Nodes: (i, "begin"), (i, s) for step s, (i, "trigger"), (i, "complete").  Returns the
    transitive closure as a dict node -> set of nodes it precedes."""
    edges = {}

    def edge(a, b):
        edges.setdefault(a, set()).add(b)
        edges.setdefault(b, set())

    for i, k in enumerate(kernels):
        prev = (i, "begin")
        edges.setdefault(prev, set())
        triggered = False
        for s, st in enumerate(k.steps):
            node = (i, s)
            edge(prev, node)
            if st[0] == "wait" and i > 0:
                edge((i - 1, "complete"), node)
            if st[0] == "trigger":
                edge(node, (i, "trigger"))
                triggered = True
            prev = node
        edge(prev, (i, "complete"))
        if not triggered:
            edge((i, "complete"), (i, "trigger"))
        if i > 0:
            edge((i - 1, "trigger") if k.pdl else (i - 1, "complete"), (i, "begin"))
    # transitive closure (the graphs are small)
    order = {n: set() for n in edges}
    for n in edges:
        stack = list(edges[n])
        while stack:
            m = stack.pop()
            if m not in order[n]:
                order[n].add(m)
                stack.extend(edges[m])
    return order


def races(kernels):
    """Pairs of accesses (kernel i before kernel j in stream order, one a write, same buffer)
    whose steps are not ordered i -> j."""
    hb = happens_before(kernels)
    acc = []
    for i, k in enumerate(kernels):
        for s, st in enumerate(k.steps):
            if st[0] in ("read", "write"):
                for buf in st[1:]:
                    acc.append((i, s, st[0], buf))
    bad = []
    for (i, s, a, x), (j, t, b, y) in itertools.combinations(acc, 2):
        if i == j or x != y or (a == "read" and b == "read"):
            continue
        if (j, t) not in hb[(i, s)]:
            bad.append((kernels[i].name, a, x, kernels[j].name, b))
    return bad


# --------------------------------------------------------------------------- the kernels

IN = ("q", "k", "v", "o", "do", "lse")


def producer():  # a kernel (torch, or the caller's) that writes the inputs
    return Kernel("producer", [("write",) + IN], pdl=False)


def consumer():  # a kernel that reads the outputs and overwrites the inputs and workspace
    return Kernel("consumer", [("read", "dq", "dk", "dv", "out", "lse_out"),
                               ("write",) + IN + ("ws", "part")], pdl=False)


def preprocess(trigger=True):
    steps = ([("trigger",)] if trigger else []) + [("read", "o", "do", "lse"), ("write", "ws")]
    return Kernel("preprocess", steps, pdl=False)


def dkv(wait=True, trigger=True):
    steps = [("wait",)] if wait else []
    steps += [("trigger",)] if trigger else []
    steps += [("read", "q", "k", "v", "do", "ws"), ("write", "dk", "dv")]
    return Kernel("dkv", steps, pdl=True)


def dq(wait_first, wait_last=True):
    steps = [("wait",)] if wait_first else []
    steps += [("read", "q", "k", "v", "do", "ws"), ("write", "dq")]
    steps += [("wait",)] if wait_last else []
    return Kernel("dq", steps, pdl=True)


def fa_bwd(**mut):
    """The fixed-length fa_bwd: dQ directly after dK/dV starts without its first wait."""
    return [preprocess(mut.get("pre_trigger", True)),
            dkv(mut.get("dkv_wait", True), mut.get("dkv_trigger", True)),
            dq(mut.get("dq_wait_first", False), mut.get("dq_wait_last", True))]


def stages(order):
    """fa_bwd_stage calls: stage 2 alone always waits first."""
    ks = {0: preprocess(), 1: dkv(), 2: dq(wait_first=True)}
    return [ks[s] for s in order]


def decode(splits=2, combine_wait=True, split_wait=True):
    split = Kernel("split", ([("wait",)] if split_wait else []) +
                   [("trigger",), ("read", "q", "k", "v"),
                    ("write",) + (("part",) if splits > 1 else ("out", "lse_out"))], pdl=True)
    ks = [split]
    if splits > 1:
        ks.append(Kernel("combine", ([("wait",)] if combine_wait else []) +
                         [("trigger",), ("read", "part"), ("write", "out", "lse_out")], pdl=True))
    return ks


# --------------------------------------------------------------------------- the library's chains

def test_fa_bwd_between_a_producer_and_a_consumer_is_ordered():
    assert races([producer()] + fa_bwd() + [consumer()]) == []


def test_two_backward_calls_on_one_workspace_are_ordered():
    assert races([producer()] + fa_bwd() + fa_bwd() + [consumer()]) == []
    assert races([producer()] + fa_bwd() + stages([0, 2, 1]) + [consumer()]) == []


@pytest.mark.parametrize("order", [(0, 1, 2), (0, 2, 1)])
def test_backward_stages_in_either_order_are_ordered(order):
    assert races([producer()] + stages(order) + [consumer()]) == []


@pytest.mark.parametrize("splits", [1, 2])
def test_decode_steps_back_to_back_are_ordered(splits):
    ks = [producer()] + decode(splits) + decode(splits) + fa_bwd() + decode(splits) + [consumer()]
    assert races(ks) == []


# --------------------------------------------------------------------------- mutations

def test_model_catches_a_dkv_that_reads_before_the_preprocess_is_done():
    bad = races([producer()] + fa_bwd(dkv_wait=False) + [consumer()])
    assert ("preprocess", "write", "ws", "dkv", "read") in bad


def test_model_catches_a_dq_that_may_complete_before_dkv():
    # without its last wait the consumer may overwrite q while dK/dV still reads it
    bad = races([producer()] + fa_bwd(dq_wait_last=False) + [consumer()])
    assert ("dkv", "read", "q", "consumer", "write") in bad


def test_model_catches_a_dq_stage_run_right_after_the_preprocess_without_its_first_wait():
    ks = [producer(), preprocess(), dq(wait_first=False)]
    assert ("preprocess", "write", "ws", "dq", "read") in races(ks + [consumer()])


def test_model_catches_a_dkv_that_triggers_before_its_wait():
    # dQ (no first wait) launched before the preprocess has completed would read its workspace
    k = Kernel("dkv", [("trigger",), ("wait",), ("read", "q", "k", "v", "do", "ws"),
                       ("write", "dk", "dv")], pdl=True)
    ks = [producer(), preprocess(), k, dq(wait_first=False), consumer()]
    assert ("preprocess", "write", "ws", "dq", "read") in races(ks)


def test_model_catches_a_combine_without_its_wait():
    bad = races([producer()] + decode(2, combine_wait=False) + [consumer()])
    assert ("split", "write", "part", "combine", "read") in bad


def test_model_catches_a_split_kernel_without_its_wait():
    # after a producer that triggers only at its end nothing can go wrong, but the next step's
    # split, begun once the combine has triggered, would overwrite the partial results the
    # combine is still reading
    assert races([producer()] + decode(2, split_wait=False) + [consumer()]) == []
    bad = races([producer()] + decode(2) + decode(2, split_wait=False) + [consumer()])
    assert ("combine", "read", "part", "split", "write") in bad
