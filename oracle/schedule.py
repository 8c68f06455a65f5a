"""Integer host logic of the path: varlen offsets, seam-window bodies, LPT order.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain Python integers.

Sources: youleyou.com HYPIC article, seam-window paragraph (the first w tokens
of each reused segment are left out of the cache) and segment-parallelism
paragraph (cold segments are dispatched with a longest-processing-time-first
greedy balance instead of round robin).

Readings where the pages are silent:
* a work item is one (segment, stream) unit; its cost is its body length in
  tokens, L_i - min(w, L_i);
* the LPT order sorts items by (-cost, segment, stream);
* the static assignment walks that order and gives each item to the worker with
  the least load so far, the lowest worker id on ties;
* item id = segment * n_streams + stream.
"""
from __future__ import annotations

import heapq


def offsets_from_lengths(lengths):
    """Exclusive prefix sum: offsets[0] = 0, offsets[i+1] = offsets[i] + L_i."""
    out = [0]
    for L in lengths:
        L = int(L)
        if L < 0:
            raise ValueError("negative segment length")
        out.append(out[-1] + L)
    return out


def validate_offsets(offsets, n_tok=None):
    """True when offsets[0] == 0, non-decreasing, and offsets[-1] == n_tok
    (when n_tok is given)."""
    offs = [int(x) for x in offsets]
    if not offs or offs[0] != 0:
        return False
    for a, b in zip(offs, offs[1:]):
        if b < a:
            return False
    if n_tok is not None and offs[-1] != int(n_tok):
        return False
    return True


def body_ranges(offsets, seam_w):
    """[(start, end)] of each segment's cached body: the first min(w, L) tokens
    are the seam window and are skipped."""
    out = []
    for a, b in zip(offsets, offsets[1:]):
        a, b = int(a), int(b)
        out.append((a + min(int(seam_w), b - a), b))
    return out


def lpt_schedule(offsets, seam_w, n_streams, n_workers):
    """Longest-processing-time-first order and greedy static assignment.

    Returns (order, worker): order is the list of item ids in LPT order;
    worker[item] is the worker that item is assigned to."""
    bodies = body_ranges(offsets, seam_w)
    items = []
    for seg, (a, b) in enumerate(bodies):
        for s in range(int(n_streams)):
            items.append((-(b - a), seg, s))
    items.sort()
    order = [seg * int(n_streams) + s for (_, seg, s) in items]
    # (load, worker id) min-heap: the least-loaded worker, lowest id on ties
    heap = [(0, w) for w in range(int(n_workers))]
    worker = [0] * len(order)
    for cost_neg, seg, s in items:
        load, best = heapq.heappop(heap)
        worker[seg * int(n_streams) + s] = best
        heapq.heappush(heap, (load - cost_neg, best))
    return order, worker


def split_pieces(offsets, seam_w, piece_tokens):
    """Pieces of a split build: each segment's seam window (when it has one) is
    a piece of its own that no segment uses, and its body is cut into pieces of
    at most ``piece_tokens`` tokens, in token order; the pieces cover all
    tokens in order.  Returns (piece_offsets, body_pieces): the offsets of the
    pieces and, per segment, the indices of its body pieces in order.

    Reading (the pages' composition law applied to a cut segment, youleyou.com
    HYPIC article, linear-layer paragraph): a body cut into consecutive pieces
    composes back to the body's pair, so only the cut itself is fixed here."""
    P = int(piece_tokens)
    if P < 1:
        raise ValueError("piece_tokens must be positive")
    out = [0]
    body = []
    for a, b in zip(offsets, offsets[1:]):
        a, b = int(a), int(b)
        w = min(int(seam_w), b - a)
        if w > 0:
            out.append(a + w)
        mine = []
        pos = a + w
        while pos < b:
            mine.append(len(out) - 1)
            pos = min(pos + P, b)
            out.append(pos)
        body.append(mine)
    return out, body
