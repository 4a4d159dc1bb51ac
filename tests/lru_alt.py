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


def replay_tokens(ctx, P, B, hot_block, resident, steps):
    """Speculative decoding: each step is a list of T top-K rows (one per
    verify token), resolved together.  A position an earlier token of the step
    also selected takes no slot of its own and reports that entry's row; a
    repeat inside one token's row is an input error.  Returns per step
    (rows[T][K], slot_pos copy, err_bits)."""
    recency = list(range(B))          # least recent first
    holder = [None] * B               # position held by each slot
    out = []
    for rows_t in steps:
        T, K = len(rows_t), len(rows_t[0])
        rows = [[-1] * K for _ in range(T)]
        err = 0
        first = {}                    # position -> (t, j) of its first entry
        later = []                    # entries that repeat another token's position
        used = set()
        pending = []
        for t in range(T):
            for j, p in enumerate(rows_t[t]):
                if p == -1:
                    continue
                if p < 0 or p >= ctx:
                    err |= 1
                    continue
                if p in first:
                    if first[p][0] == t:
                        err |= 2
                    else:
                        later.append((t, j, first[p]))
                    continue
                first[p] = (t, j)
                page = p // P
                if page in resident:
                    rows[t][j] = resident[page] * P + p % P
                    continue
                if p in holder:
                    s = holder.index(p)
                    used.add(s)
                    rows[t][j] = hot_block[s // P] * P + s % P
                    continue
                pending.append((t, j))
        for (t, j) in pending:
            victim = next((s for s in recency if s not in used), None)
            if victim is None:
                err |= 4
                continue
            used.add(victim)
            holder[victim] = rows_t[t][j]
            rows[t][j] = hot_block[victim // P] * P + victim % P
        for (t, j, (t0, j0)) in later:
            rows[t][j] = rows[t0][j0]
        recency = [s for s in recency if s not in used] + sorted(used)
        out.append((rows, [(-1 if h is None else h) for h in holder], err))
    return out
