"""The fragment-lookup oracle against the behaviour the blend-index page states (sections 三, 四, 六, 七)
and the algebra of a polynomial hash.  Each check also runs against planted mistakes."""
import random

import pytest

import oracle.matcher as om

C = 16


def _toks(rng, n, vocab=50000):
    return [rng.randrange(vocab) for _ in range(n)]


def check_fingerprint_algebra(m):
    """A single token hashes to itself, two tokens to a*B + b, and the window hash rolls:
    H(i+1) = (H(i) - t_i B^(C-1)) B + t_(i+C)  (mod 2^64)."""
    assert m.fingerprint([7]) == 7
    assert m.fingerprint([3, 5]) == (3 * om.POLY_BASE + 5) % (1 << 64)
    rng = random.Random(1)
    t = _toks(rng, 200, 1 << 32)
    top = pow(om.POLY_BASE, C - 1, 1 << 64)
    for i in range(0, 200 - C):
        h0, h1 = m.fingerprint(t[i:i + C]), m.fingerprint(t[i + 1:i + 1 + C])
        assert h1 == ((h0 - t[i] * top) * om.POLY_BASE + t[i + C]) % (1 << 64)


def check_planted_and_near_miss(m):
    """A stored chunk is found where it sits in the request (old_st from the index, cur_st from the
    request); a window differing in one token is rejected."""
    rng = random.Random(2)
    idx = m.BlendIndex(C)
    a, b = _toks(rng, C), _toks(rng, C)
    idx.add(a, occ_id=10, old_st=512, ns=1)
    idx.add(b, occ_id=11, old_st=0, ns=1)
    near = list(b)
    near[5] += 1
    q = _toks(rng, 40) + a + _toks(rng, 7) + near + _toks(rng, 3)
    assert idx.match(q, ns=1) == [(10, 512, 40)]


def check_namespaces(m):
    """A content claimed only by another namespace is not returned; one claimed by several is returned
    to each with its own occupant."""
    rng = random.Random(3)
    idx = m.BlendIndex(C)
    a = _toks(rng, C)
    idx.add(a, occ_id=1, old_st=0, ns=2)
    q = _toks(rng, 9) + a
    assert idx.match(q, ns=1) == []
    idx.add(a, occ_id=2, old_st=64, ns=1)
    assert idx.match(q, ns=1) == [(2, 64, 9)]
    assert idx.match(q, ns=2) == [(1, 0, 9)]


def check_two_prefixes_survive_one_eviction(m):
    """The same content stored under two chunks (two prefixes) in one namespace: both are matchable, in
    first-indexing order, at most one match each; removing one leaves the other discoverable."""
    rng = random.Random(4)
    idx = m.BlendIndex(C)
    a = _toks(rng, C)
    idx.add(a, occ_id=5, old_st=0, ns=1)
    idx.add(a, occ_id=6, old_st=128, ns=1)
    q = a + _toks(rng, 5) + a + _toks(rng, 2) + a
    assert idx.match(q, ns=1) == [(5, 0, 0), (6, 128, C + 5)]
    idx.remove(5)
    assert idx.match(q, ns=1) == [(6, 128, 0)]


def check_collision_never_added(m, monkeypatch=None):
    """A second content under an existing fingerprint is never added, so it is never matched (here with
    a deliberately weak hash to force the collision)."""
    rng = random.Random(5)
    weak = lambda toks: sum(int(t) for t in toks) % 7
    saved = m.fingerprint
    m.fingerprint = weak
    try:
        idx = m.BlendIndex(C)
        a = _toks(rng, C)
        b = list(a)
        b[0], b[1] = b[1], b[0]                   # same sum, different content
        if a == b:
            b[0] += 7
            b[1] -= 7
        assert idx.add(a, 1, 0, 1) is True
        assert idx.add(b, 2, 0, 1) is False
        assert idx.match(_toks(rng, 3) + b, ns=1) == []
        assert idx.match(_toks(rng, 3) + a, ns=1) == [(1, 0, 3)]
    finally:
        m.fingerprint = saved


def check_index_rules(m):
    """Unknown stored position (old_st -1) and wrong-length chunks are not indexed; probing every s-th
    position finds only aligned chunks."""
    rng = random.Random(6)
    idx = m.BlendIndex(C)
    a, b = _toks(rng, C), _toks(rng, C)
    assert idx.add(a, 1, -1, 1) is False
    assert idx.add(a[:-1], 2, 0, 1) is False
    assert idx.add(b, 3, 0, 1) is True
    assert idx.match(_toks(rng, 4) + a, ns=1) == []
    assert idx.match(_toks(rng, 3) + b, ns=1, stride=2) == []
    assert idx.match(_toks(rng, 4) + b, ns=1, stride=2) == [(3, 0, 4)]


def check_leftmost_greedy(m):
    """Overlapping matches: the earlier one wins; touching matches are both kept."""
    ms = [(2, 0, 8), (1, 0, 0), (3, 0, 16), (4, 0, 31), (5, 0, 40)]
    assert m.leftmost_greedy(ms, C) == [(1, 0, 0), (3, 0, 16), (5, 0, 40)]
    # a chain where keeping the later of two overlapping matches would keep a different set
    assert m.leftmost_greedy([(1, 0, 0), (2, 0, 10), (3, 0, 26)], C) == [(1, 0, 0), (3, 0, 26)]


CHECKS = [check_fingerprint_algebra, check_planted_and_near_miss, check_namespaces,
          check_two_prefixes_survive_one_eviction, check_collision_never_added, check_index_rules,
          check_leftmost_greedy]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_matcher_oracle(check):
    check(om)


def _fp_reversed(tokens):
    h = 0
    for t in reversed(list(tokens)):
        h = (h * om.POLY_BASE + (int(t) & 0xFFFFFFFF)) & om.MASK64
    return h


def _greedy_later_wins(matches, chunk_size):
    kept, start = [], 1 << 62
    for mt in sorted(matches, key=lambda x: -x[2]):
        if mt[2] + chunk_size <= start:
            kept.append(mt)
            start = mt[2]
    return sorted(kept, key=lambda x: x[2])


class _FirstOccupantOnly(om.BlendIndex):
    def match(self, tokens, ns, stride=1):
        # ignores the namespace when choosing the occupant
        out, seen, C = [], set(), self.C
        tokens = [int(t) & 0xFFFFFFFF for t in tokens]
        for i in range(0, len(tokens) - C + 1, stride):
            e = self.contents.get(om.fingerprint(tuple(tokens[i:i + C])))
            if e and tuple(tokens[i:i + C]) == e["tokens"]:
                o = e["occupants"][0]
                if o[0] not in seen:
                    out.append((o[0], o[1], i))
                    seen.add(o[0])
        return out


@pytest.mark.parametrize("name,bad", [("fingerprint", _fp_reversed), ("leftmost_greedy", _greedy_later_wins),
                                      ("BlendIndex", _FirstOccupantOnly)], ids=["fp_reversed", "later_wins",
                                                                                "ignores_namespace"])
def test_matcher_pins_catch_mutation(monkeypatch, name, bad):
    monkeypatch.setattr(om, name, bad)
    caught = 0
    for check in CHECKS:
        try:
            check(om)
        except Exception:
            caught += 1
    assert caught, f"no pin caught {bad.__name__}"
