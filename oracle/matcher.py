"""CPU oracle of the CacheBlend fragment lookup (TEST INFRASTRUCTURE ONLY; plain Python integers).

Source: the LMCache coordinator blend-index page (nxmr.cn/news/96227), sections "三、身份与作用域"
(content fingerprint, namespaces), "四、数据结构与召回" (the two-level structure and the match flow:
filter, resolve, choose the requester's occupant, verify tokens, mark seen), "六、HTTP 接口" (matches
(chunk, old_st, cur_st) ascending by cur_st, at most one per chunk, overlaps resolved by the caller with
leftmost-greedy) and "七" (the blend keeps the earlier of two overlapping matches).

Readings where the pages leave a step open:
  M1  fingerprint of a window t_0..t_{C-1}: Horner's rule h = h * B + t_j over the tokens in order,
      modulo 2^64, tokens as unsigned 32-bit values, B = 0x9E3779B97F4A7C15 (the page's fleet constant).
  M2  a fingerprint names one content: the first content stored under it; a different content with the
      same fingerprint is never added (it stays undiscoverable, never mismatched).
  M3  a content's occupants keep their first-indexing order; a window that verifies is given the first
      occupant claimed by the requester's namespace whose chunk has not matched yet.
  M4  windows are probed at positions 0, s, 2s, ... (s = probe stride) while a whole window fits.
  M5  leftmost-greedy: matches sorted by cur_st; one is kept when it starts at or after the end of the
      last kept one.
The occupancy filter of the page only skips dictionary lookups that would fail; it cannot change a
result, so the oracle resolves every window in the dictionary directly.
"""
from __future__ import annotations

POLY_BASE = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1


def fingerprint(tokens) -> int:
    """Reading M1: Horner's rule modulo 2^64."""
    h = 0
    for t in tokens:
        h = (h * POLY_BASE + (int(t) & 0xFFFFFFFF)) & MASK64
    return h


class BlendIndex:
    """Content entries keyed by fingerprint; each holds the content's tokens and its occupants
    (occupant id, old_st, namespace) in first-indexing order."""

    def __init__(self, chunk_size: int):
        self.C = chunk_size
        self.contents = {}       # fingerprint -> {"tokens": tuple, "occupants": [(id, old_st, ns), ...]}

    def add(self, tokens, occ_id: int, old_st: int, ns: int) -> bool:
        """Index one stored chunk.  Returns False when it is not indexed: wrong length, unknown position
        (old_st < 0: the page's UNKNOWN_TOKEN_OFFSET), or a fingerprint already naming other content."""
        tokens = tuple(int(t) & 0xFFFFFFFF for t in tokens)
        if len(tokens) != self.C or old_st < 0:
            return False
        fp = fingerprint(tokens)
        e = self.contents.get(fp)
        if e is None:
            self.contents[fp] = {"tokens": tokens, "occupants": [(occ_id, old_st, ns)]}
            return True
        if e["tokens"] != tokens:
            return False                          # M2
        e["occupants"].append((occ_id, old_st, ns))
        return True

    def remove(self, occ_id: int) -> None:
        """Drop an occupant (the page's claim removal); a content without occupants is dropped."""
        for fp in list(self.contents):
            e = self.contents[fp]
            e["occupants"] = [o for o in e["occupants"] if o[0] != occ_id]
            if not e["occupants"]:
                del self.contents[fp]

    def match(self, tokens, ns: int, stride: int = 1) -> list:
        """All matches (occ_id, old_st, cur_st), ascending cur_st, at most one per occupant."""
        tokens = [int(t) & 0xFFFFFFFF for t in tokens]
        C, out, seen = self.C, [], set()
        for i in range(0, len(tokens) - C + 1, stride):
            window = tuple(tokens[i:i + C])
            e = self.contents.get(fingerprint(window))
            if e is None:
                continue
            cand = [o for o in e["occupants"] if o[2] == ns and o[0] not in seen]
            if not cand:
                continue                          # nothing this requester may use: no comparison
            if window != e["tokens"]:
                continue                          # verification
            occ_id, old_st, _ = cand[0]
            out.append((occ_id, old_st, i))
            seen.add(occ_id)                      # marked only after verification
        return out


def leftmost_greedy(matches, chunk_size: int) -> list:
    """Reading M5: keep matches in cur_st order that do not overlap an earlier kept one."""
    kept, end = [], -1
    for m in sorted(matches, key=lambda m: m[2]):
        if m[2] >= end:
            kept.append(m)
            end = m[2] + chunk_size
    return kept
