"""Source checks on the CUDA kernels that need no GPU.

A full-mask warp collective (``__shfl_sync(0xffffffff, ...)``, ``__any_sync``,
``__reduce_*_sync``, ``__match_any_sync``, ``__syncwarp``) must be reached by
all 32 lanes of the warp, and ``__syncthreads`` by every thread of the block.
A loop whose start depends on the lane or the thread index
(``for (int v = lane; v < n; v += 32)``) runs a different number of times on
different lanes once ``n`` is not a multiple of the stride. A collective inside
such a loop then waits on lanes that have left it. The kernel hangs as soon as
a warp goes round its outer loop a second time, because the lanes that left
the inner loop reach a different collective.

These tests parse the kernel sources and fail if any loop of that shape holds
a collective. Such loops must step warp-uniformly instead
(``for (int v0 = 0; v0 < n; v0 += 32) { const int v = v0 + lane; ... }``).
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "combine_router_gemm_top_b300", "csrc")

# a loop init or bound that differs between lanes or threads of one warp;
# the warp's index (threadIdx.x >> 5, / 32, & ~31) is the same on all lanes
_LANE_DEPENDENT = re.compile(r"\blane\b|threadIdx\.x")
_WARP_UNIFORM = re.compile(
    r"\(?\s*threadIdx\.x\s*(>>\s*5|/\s*32|&\s*~\s*31)\s*\)?")
_COLLECTIVE = re.compile(
    r"__(shfl|shfl_up|shfl_down|shfl_xor|any|all|ballot|match_any|"
    r"reduce_(add|min|max|and|or|xor))_sync\s*\(|__syncwarp\s*\(|"
    r"__syncthreads\s*\(|\bwarp_(sum|min|max)\w*\s*\(|\bbwd_warp_sum\s*\(|"
    r"\bwarp_sum_f32\s*\(")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cuh")))


def _strip_comments(text):
    text = re.sub(r"/\*.*?\*/", lambda m: re.sub(r"[^\n]", " ", m.group()),
                  text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def _matching(text, i, open_ch, close_ch):
    """Index just past the bracket that closes the one at text[i]."""
    depth = 0
    for j in range(i, len(text)):
        if text[j] == open_ch:
            depth += 1
        elif text[j] == close_ch:
            depth -= 1
            if depth == 0:
                return j + 1
    raise ValueError("unbalanced brackets")


def lane_strided_loops(text):
    """(line, header, body) of every for loop whose init or condition
    depends on the lane or thread index."""
    text = _strip_comments(text)
    out = []
    for m in re.finditer(r"\bfor\s*\(", text):
        h0 = m.end() - 1
        h1 = _matching(text, h0, "(", ")")
        header = text[h0 + 1:h1 - 1]
        parts = header.split(";")
        if len(parts) != 3:
            continue   # a range-for or a macro: not the pattern
        init, cond = (_WARP_UNIFORM.sub(" w ", p) for p in parts[:2])
        if not (_LANE_DEPENDENT.search(init) or _LANE_DEPENDENT.search(cond)):
            continue
        k = h1
        while k < len(text) and text[k].isspace():
            k += 1
        if k < len(text) and text[k] == "{":
            body = text[k:_matching(text, k, "{", "}")]
        else:
            body = text[k:text.index(";", k) + 1]
        out.append((text.count("\n", 0, m.start()) + 1, header.strip(), body))
    return out


@pytest.mark.parametrize("path", _sources(), ids=os.path.basename)
def test_no_collective_in_lane_dependent_loop(path):
    with open(path) as f:
        loops = lane_strided_loops(f.read())
    bad = [f"{os.path.basename(path)}:{line}: for ({hdr}) holds "
           f"{_COLLECTIVE.search(body).group().strip()}"
           for line, hdr, body in loops if _COLLECTIVE.search(body)]
    assert not bad, "\n".join(bad)


def test_checker_flags_the_divergent_form():
    """The checker itself: the form that hung is flagged, the warp-uniform
    form that replaced it is not, and a collective after the loop is fine."""
    divergent = """
    for (int v0 = v_begin + lane; v0 < v_end; v0 += 128) {
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_dst, j);
      }
    }"""
    uniform = """
    for (int v0 = v_begin; v0 < v_end; v0 += 128) {
      const int v = v0 + lane;
      const int r = __shfl_sync(0xffffffffu, my_dst, 0);
    }"""
    after = """
    for (int d = lane; d < D; d += 32) acc += x[d];
    acc = warp_sum_f32(acc);"""
    block = """
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      s[i] = 0;
      __syncthreads();
    }"""
    per_warp = """
    for (int64_t q0 = lo + (threadIdx.x & ~31); q0 < hi; q0 += blockDim.x) {
      const unsigned peers = __match_any_sync(0xffffffffu, d);
    }"""
    flagged = lambda src: any(_COLLECTIVE.search(b)
                              for _, _, b in lane_strided_loops(src))
    assert flagged(divergent)
    assert not flagged(uniform)
    assert not flagged(after)
    assert flagged(block)
    assert not flagged(per_warp)
