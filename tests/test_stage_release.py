"""Source check of the stage reuse protocol of the staged kernels (no GPU).

A consumer thread of a staged kernel reads a shared-memory stage with plain
loads and then releases it (arrive on the stage's "empty" barrier), after which
the producer refills it with bulk copies.  Release/acquire on the barrier does
not order the consumer's generic-proxy loads before the refill's async-proxy
writes, so the kernels rely on a data dependency instead: every consumer arrive
comes after global stores that consume what the thread loaded from the stage.
This test reads csrc/kernels_tma.cu and checks, for every consumer-side arrive
on an empty barrier, that between the wait on the matching "full" barrier and
the arrive every shared-memory load of the stage is followed by a global store.
It also checks that the arrive and the wait carry their semantics explicitly.
"""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "fsdp_sharded_optimizer_flatparameter_gb300", "csrc", "kernels_tma.cu")

# the staged kernels' consumer code (k_fused_tma's lives in fused_tma_body, k_rs_tma's / k_ar_tma's in
# rs_tma_body and k_dp_tma's in dp_tma_body, which the kernels call)
KERNELS = ("fused_tma_body", "k_fused_tma_list", "rs_tma_body", "dp_tma_body")
LOAD = re.compile(r"\blds_(?:bf|f32)<")
STORE = re.compile(r"\b__stcs\(|\bstg_f32<")
# consumer releases: empty[...] pairs with full[...], gempty[...] with gfull[...]
ARRIVE = re.compile(r"mbar_arrive\(&(empty|gempty)\[")
PAIR = {"empty": "full", "gempty": "gfull"}


def _strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def _kernel_body(text, name):
    m = re.search(r"(?:__global__|__device__)[^\n]*\bvoid[^\n]*\b%s\(" % re.escape(name), text)
    assert m, "kernel %s not found" % name
    start = text.index("{", m.end())
    depth, i = 0, start
    while True:
        c = text[i]
        if c == "{":
            depth += 1
        elif c == "}":
            depth -= 1
            if depth == 0:
                return text[start:i + 1]
        i += 1


def _consumer_part(body):
    # the producer is the `if (warp == 0) { ... return; }` block; consumers follow it
    m = re.search(r"if \(warp == 0\) \{", body)
    assert m
    depth, i = 0, body.index("{", m.start())
    while True:
        if body[i] == "{":
            depth += 1
        elif body[i] == "}":
            depth -= 1
            if depth == 0:
                return body[i + 1:]
        i += 1


def test_every_consumer_arrive_follows_the_stores_that_consume_the_stage():
    text = _strip_comments(open(SRC).read())
    checked = 0
    for name in KERNELS:
        cons = _consumer_part(_kernel_body(text, name))
        arrives = list(ARRIVE.finditer(cons))
        assert arrives, "%s: no consumer arrive found" % name
        for a in arrives:
            full = PAIR[a.group(1)]
            waits = [w.start() for w in re.finditer(r"mbar_wait\(&%s\[" % full, cons) if w.start() < a.start()]
            assert waits, "%s: arrive on %s without a preceding wait on %s" % (name, a.group(1), full)
            span = cons[waits[-1]:a.start()]
            loads = [m.end() for m in LOAD.finditer(span)]
            if not loads:
                continue
            stores = [m.start() for m in STORE.finditer(span)]
            assert stores and max(stores) > max(loads), (
                "%s: an arrive on %s[] releases a stage whose loads no global store after them consumes"
                % (name, a.group(1)))
            checked += 1
    assert checked >= 6
    assert "fused_tma_body<" in _kernel_body(text, "k_fused_tma")
    assert "rs_tma_body<" in _kernel_body(text, "k_rs_tma") and "rs_tma_body<" in _kernel_body(text, "k_ar_tma")
    assert "dp_tma_body<" in _kernel_body(text, "k_dp_tma")


def test_barrier_semantics_are_explicit():
    text = open(SRC).read()
    assert "mbarrier.arrive.release.cta.shared::cta.b64" in text
    assert "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64" in text
    assert not re.search(r"mbarrier\.arrive\.shared::cta", text)
    assert not re.search(r"mbarrier\.try_wait\.parity\.shared::cta", text)


def test_the_check_catches_an_early_release():
    """A planted early release (arrive right after the loads) must fail the rule above."""
    body = _strip_comments(open(SRC).read())
    cons = _consumer_part(_kernel_body(body, "rs_tma_body"))
    early = cons.replace("lds_bf<VPT>(sg + (size_t)q * T + e, f);",
                         "lds_bf<VPT>(sg + (size_t)q * T + e, f); mbar_arrive(&empty[s]);", 1)
    assert early != cons
    a = next(ARRIVE.finditer(early))
    span = early[[w.start() for w in re.finditer(r"mbar_wait\(&full\[", early) if w.start() < a.start()][-1]:a.start()]
    loads = [m.end() for m in LOAD.finditer(span)]
    stores = [m.start() for m in STORE.finditer(span)]
    assert loads and not (stores and max(stores) > max(loads))
