"""Oracle of the n-gram drafting rule of speculative decoding.

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` alone; no code shared with
the library.

kimi-k3-in-c k3_run.c, ``spec_draft`` (the function's own statement of its
rule): drafts are proposals read from the sequence itself.  For a suffix
length n of 4, then 3, look for earlier occurrences of the sequence's last n
ids; from the most recent one, propose the ids that followed it, at most
``cap`` (8 at most) and never past the end of the sequence.  When the suffix
occurred at least twice, the two most recent occurrences must agree: the
draft ends at the first position where their continuations differ, or where
the older continuation would run into the newer occurrence.  The first n
with a non-empty draft is used; none gives no draft.  (The page's header
comment for --spec says "3, then 2"; the function's statement, which also
explains why eager drafts were dropped, says 4 then 3 with the agreement
rule; the latter is followed.)
"""


def spec_draft(seq, cap=8):
    seq = [int(t) for t in seq]
    cap = min(int(cap), 8)
    T = len(seq)
    if cap < 1:
        return []
    for n in (4, 3):
        if T < n + 1:
            continue
        suffix = seq[T - n:]
        starts = [j for j in range(T - n - 1, -1, -1) if seq[j:j + n] == suffix][:2]
        if not starts:
            continue
        newest = starts[0]
        older = starts[1] if len(starts) > 1 else None
        draft = []
        for i in range(cap):
            k = newest + n + i
            if k >= T:
                break
            if older is not None and (older + n + i >= newest or seq[older + n + i] != seq[k]):
                break
            draft.append(seq[k])
        if draft:
            return draft
    return []
