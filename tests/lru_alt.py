"""A second, independently written model of RESOLVE's hot buffer, for pinning
the oracle on tiny traces.  Test helper only.

Where the oracle keeps per-slot stamps and sorts victim candidates, this model
keeps one recency list of slots (least recent first).  Slots used in a step
are pinned for that step; after the step every used slot moves to the
most-recent end, lower slot numbers first (several slots used in one step are
equally recent, and the lower slot counts as older).  Empty slots start at the
least-recent end in slot order.  Resident positions bypass the buffer.
"""


def replay(ctx, P, B, hot_block, resident, steps):
    """resident: {page: block}; steps: list of top-K lists.
    Returns per step (rows, slot_pos copy, err_bits)."""
    recency = list(range(B))          # least recent first
    holder = [None] * B               # position held by each slot
    out = []
    for topk in steps:
        rows = [-1] * len(topk)
        err = 0
        seen = set()
        used = set()
        pending = []
        for j, p in enumerate(topk):
            if p == -1:
                continue
            if p < 0 or p >= ctx:
                err |= 1
                continue
            if p in seen:
                err |= 2
                continue
            seen.add(p)
            page = p // P
            if page in resident:
                rows[j] = resident[page] * P + p % P
                continue
            if p in holder:
                s = holder.index(p)
                used.add(s)
                rows[j] = hot_block[s // P] * P + s % P
                continue
            pending.append(j)
        for j in pending:
            victim = next((s for s in recency if s not in used), None)
            if victim is None:
                err |= 4
                continue
            used.add(victim)
            holder[victim] = topk[j]
            rows[j] = hot_block[victim // P] * P + victim % P
        recency = [s for s in recency if s not in used] + sorted(used)
        out.append((rows, [(-1 if h is None else h) for h in holder], err))
    return out
