"""tcgen05 fence lint: a static check, on the CPU, of how the library's CUDA sources order their
tensor-core (tcgen05) operations against thread synchronisation.

tcgen05 operations run asynchronously to the issuing thread, so a barrier or an mbarrier wait
alone does not order them between threads.  PTX requires, around every synchronisation that
hands tensor memory (its contents, or its address) from one thread to another:
  - in the thread that produced it (a tcgen05.ld that must finish before the memory is
    overwritten, an allocation whose address it wrote): tcgen05.fence::before_thread_sync
    before the synchronisation;
  - in the thread that consumes it (a tcgen05.ld, an MMA issue, a deallocation, a read of the
    allocated address): tcgen05.fence::after_thread_sync after the synchronisation.
A tcgen05.commit carries the "before" fence implicitly, so a wait on the mbarrier that a commit
arrives on needs only the "after" fence.  Operands that threads write to shared memory with
ordinary stores must also cross into the async proxy (fence.proxy.async) before an MMA reads
them.

Rules, checked over each kernel body in source order (loops are read as straight-line text; a
loop body that hands tensor memory to its next iteration is fenced inside the body):
  R1  every consumer (TMEM load, MMA issue, deallocation, read of the allocated address) has a
      fence_after_sync with no synchronisation point between it and the consumer;
  R2  between a TMEM load or an allocation and the next consumer there is a fence_before_sync
      followed by a synchronisation point;
  R3  every MMA issue has a fence_smem_to_async before the synchronisation that precedes it,
      and after the previous round of MMA issues.
The wait helper that ends in fence_after_sync counts as a synchronisation followed by the
fence (the lint checks that its body does end so).

The kernels of the KDA prefill use these operations; the decode / verify kernels do not.
"""
from __future__ import annotations

import glob
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "verify_kda_decode_gb300", "csrc")

# event kinds
SYNC, AFTER, BEFORE, PROXY, LD, MMA, ALLOC, DEALLOC, ADDR, WAIT_FENCED = (
    "sync", "after", "before", "proxy", "ld", "mma", "alloc", "dealloc", "addr", "wait_fenced")

PATTERNS = [
    (SYNC, r"__syncthreads\s*\(|__syncthreads_or\s*\(|mbar_wait_bounded\s*\("),
    (WAIT_FENCED, r"\bwait_all2?\s*\("),
    (AFTER, r"fence_after_sync\s*\("),
    (BEFORE, r"fence_before_sync\s*\("),
    (PROXY, r"fence_smem_to_async\s*\("),
    (LD, r"\btc::ld(?:16|32)\s*\(|\bld(?:32)?_cat\s*\("),
    (MMA, r"\btc::mma_(?:tiles|split3)(?:_bmn|_bcat|_kcat)?(?:_ks)?\s*\("),
    (ALLOC, r"\btc::tmem_alloc\s*\("),
    (DEALLOC, r"\btc::tmem_dealloc\s*\("),
    (ADDR, r"=\s*sm\.tmem\b"),
]
CONSUMERS = {LD, MMA, DEALLOC, ADDR}


def strip_comments(src: str) -> str:
    src = re.sub(r"/\*.*?\*/", lambda m: "\n" * m.group(0).count("\n"), src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def function_bodies(src: str, head: str):
    """(name, body, first line) of every function whose declaration matches `head`."""
    out = []
    for m in re.finditer(head, src):
        open_at = src.index("{", m.end())
        depth, i = 0, open_at
        while True:
            if src[i] == "{":
                depth += 1
            elif src[i] == "}":
                depth -= 1
                if depth == 0:
                    break
            i += 1
        names = [n for n in re.findall(r"(\w+)\s*\(", src[m.start():open_at]) if n != "__launch_bounds__"]
        out.append((names[0] if names else "?", src[open_at:i + 1], src.count("\n", 0, open_at) + 1))
    return out


def events(body: str, line0: int):
    ev = []
    for kind, pat in PATTERNS:
        for m in re.finditer(pat, body):
            ev.append((m.start(), kind, line0 + body.count("\n", 0, m.start())))
    ev.sort()
    return [(k, ln) for _, k, ln in ev]


def wait_helper_is_fenced(src: str) -> bool:
    """The helper `wait_all` counts as a fenced wait only if its body synchronises and then
    issues fence_after_sync before returning success."""
    bodies = function_bodies(src, r"\bbool\s+wait_all2?\s*\(")
    if not bodies:
        return False
    for _, body, _ in bodies:
        s, a = body.find("__syncthreads_or"), body.rfind("fence_after_sync")
        if not 0 <= s < a:
            return False
    return True


def lint_source(src: str, fname: str = "<src>"):
    """Violations of R1-R3 in one translation unit, as (file, line, rule, message)."""
    src = strip_comments(src)
    fenced_wait = wait_helper_is_fenced(src)
    problems = []
    for name, body, line0 in function_bodies(src, r"__global__\s+void[^;{]*?\b\w+\s*\("):
        ev = events(body, line0)
        if not any(k in CONSUMERS or k == ALLOC for k, _ in ev):
            continue
        if any(k == WAIT_FENCED for k, _ in ev) and not fenced_wait:
            problems.append((fname, line0, "R1", f"{name}: wait_all is used but does not end in fence_after_sync"))
        # R1: the last synchronisation-related event before each consumer is an "after" fence
        last = None
        for k, ln in ev:
            if k in (SYNC, AFTER, WAIT_FENCED):
                last = k
            elif k in CONSUMERS and last == SYNC:
                problems.append((fname, ln, "R1", f"{name}: {k} follows a synchronisation without fence_after_sync"))
        # R2: a load / allocation is handed on only through fence_before_sync + synchronisation
        pending = None          # (kind, line) of a load / allocation not yet handed on
        seen_before = False
        for k, ln in ev:
            if k in (LD, ALLOC):
                if pending is None:
                    pending, seen_before = (k, ln), False
                continue
            if pending is None:
                continue
            if k == BEFORE:
                seen_before = True
            elif k in (SYNC, WAIT_FENCED) and seen_before:
                pending = None
            elif k in CONSUMERS:
                problems.append((fname, pending[1], "R2", f"{name}: {pending[0]} reaches the {k} at line {ln} "
                                                          "without fence_before_sync + synchronisation"))
                pending = None
        # R3: shared-memory operands cross into the async proxy before the synchronisation that
        # hands them to the MMA issuer; MMAs issued back to back share one crossing, and a
        # synchronisation after an MMA starts a new round that needs its own
        proxied = crossed = mma_since_sync = False
        for k, ln in ev:
            if k == PROXY:
                proxied = True
            elif k in (SYNC, WAIT_FENCED):
                crossed = proxied if mma_since_sync else (crossed or proxied)
                proxied = mma_since_sync = False
            elif k == MMA:
                if not crossed:
                    problems.append((fname, ln, "R3", f"{name}: MMA issue without fence_smem_to_async before "
                                                      "the synchronisation that precedes it"))
                mma_since_sync = True
    return problems


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def test_sources_with_tensor_core_kernels_exist():
    used = [f for f in sources() if re.search(r"\btc::mma_", strip_comments(open(f).read()))]
    assert used, "no translation unit issues tcgen05 MMAs: the lint would check nothing"


@pytest.mark.parametrize("path", sources(), ids=os.path.basename)
def test_tcgen05_fences(path):
    problems = lint_source(open(path).read(), os.path.basename(path))
    assert not problems, "\n".join(f"{f}:{ln}: {r} {msg}" for f, ln, r, msg in problems)


# --------------------------------------------------------------------------- negative controls

def _prefill_src():
    return open(os.path.join(CSRC, "kda_prefill.cu")).read()


def _remove_before(src: str, needle: str, context: str) -> str:
    """src without the last `needle` that precedes the (unique) `context`."""
    assert src.count(context) == 1, context
    idx = src.rindex(needle, 0, src.index(context))
    return src[:idx] + src[idx + len(needle):]


# Planted mistakes: one fence removed where the handover it guards is real.
PLANTED = [
    # prep: the allocated address, written by warp 0, read by every thread
    ("tc::fence_before_sync();", "const uint32_t tmem = sm.tmem;", "R2"),
    ("tc::fence_after_sync();", "const uint32_t tmem = sm.tmem;", "R1"),
    # prep: the X read-out loads of every warp, then the deallocation by warp 0
    ("tc::fence_before_sync();", "tc::tmem_dealloc(tmem, 256)", "R2"),
    ("tc::fence_after_sync();", "tc::tmem_dealloc(tmem, 256)", "R1"),
    # prep: the R and T operands written by ordinary stores, then the X products
    ("tc::fence_smem_to_async();", "tc::mma_split3_kcat(tmem, smem_u32(rt)", "R3"),
    # scan: the allocated address; the W S loads of lane quarters 0, 1 before the MMA that accumulates
    # onto the same tensor memory; the deallocation after the last chunk
    ("tc::fence_after_sync();", "const uint32_t tmem = sm.tmem, d2", "R1"),
    ("tc::fence_before_sync();", "tc::mma_split3_bcat(d2,", "R2"),
    ("tc::fence_after_sync();", "tc::mma_split3_bcat(d2,", "R1"),
    ("tc::fence_smem_to_async();", "tc::mma_split3_bcat(d2,", "R3"),
    ("tc::fence_after_sync();", "tc::tmem_dealloc(tmem, kScanTmemCols)", "R1"),
]


@pytest.mark.parametrize("needle,context,rule", PLANTED)
def test_lint_catches_planted_missing_fence(needle, context, rule):
    """Each planted mistake (on a copy of the text, never on the build) fails the matching rule."""
    src = strip_comments(_prefill_src())
    assert not lint_source(src)
    problems = lint_source(_remove_before(src, needle, context))
    assert any(r == rule for _, _, r, _ in problems), (needle, context, problems)


def test_lint_requires_the_wait_helper_to_fence():
    src = strip_comments(_prefill_src())
    helper = function_bodies(src, r"\bbool\s+wait_all\s*\(")[0][1]
    broken = src.replace(helper, helper.replace("tc::fence_after_sync();", ""))
    assert any(r == "R1" for _, _, r, _ in lint_source(broken))
