"""GPU fragment matcher (cb_index_*) against the oracle of the blend-index page's lookup, bit for bit
(integer work): a 32K-token request assembled from indexed chunks of two namespaces, duplicated content
under two occupants, near misses, unindexed chunks, overlapping matches and random filler."""
import numpy as np
import pytest

import oracle.matcher as om
import workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

C = 256
VOCAB = 128256


@pytest.fixture(scope="module")
def cb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import cacheblend_selective_kv_gb300 as cbm
    return cbm


def build_case(seed=7, n_chunks=600, n_tokens=32768):
    """Indexed chunks and a request (the recipe is seeded and synthetic)."""
    rng = np.random.default_rng(seed)
    chunks = np.stack([workload.tokens(seed, 1000 + i, C, VOCAB) for i in range(n_chunks)]).astype(np.uint32)
    occ = np.arange(100, 100 + n_chunks, dtype=np.int32)
    old = (rng.integers(0, 64, n_chunks) * C).astype(np.int32)
    ns = rng.integers(1, 3, n_chunks).astype(np.int32)
    old[::37] = -1                                       # stored position unknown: not indexed
    # same content under a second occupant (another prefix) in the same namespace, and in the other one
    extra_t, extra_o, extra_s, extra_n = [], [], [], []
    for k, i in enumerate(range(5, n_chunks, 53)):
        extra_t.append(chunks[i]); extra_o.append(5000 + k); extra_s.append(7 * C); extra_n.append(ns[i])
        extra_t.append(chunks[i]); extra_o.append(6000 + k); extra_s.append(3 * C); extra_n.append(3 - ns[i])
    # a chunk that overlaps another: B = A[128:] + X[:128], so planting A then X makes B verify at +128
    a, x = 11, 12
    b = np.concatenate([chunks[a][128:], chunks[x][:128]])
    extra_t.append(b); extra_o.append(7000); extra_s.append(0); extra_n.append(ns[a])
    all_t = np.concatenate([chunks, np.stack(extra_t)])
    all_o = np.concatenate([occ, np.array(extra_o, np.int32)])
    all_s = np.concatenate([old, np.array(extra_s, np.int32)])
    all_n = np.concatenate([ns, np.array(extra_n, np.int32)])
    # request: random filler with planted chunks (some twice), near misses, and A followed by X
    req = workload.tokens(seed, 1, n_tokens, VOCAB).astype(np.int64)
    pos = 0
    plant = list(rng.permutation(n_chunks)[:90]) + [5, 5, 58, 58]
    for i in plant:
        pos += int(rng.integers(0, 300))
        if pos + C > n_tokens - 3 * C:
            break
        t = chunks[i].copy()
        if rng.random() < 0.1:
            t[int(rng.integers(0, C))] ^= 1              # near miss
        req[pos:pos + C] = t
        pos += C
    req[n_tokens - 3 * C: n_tokens - 2 * C] = chunks[a]
    req[n_tokens - 2 * C: n_tokens - C] = chunks[x]
    if ns[x] != ns[a]:
        all_n[x] = ns[a]
    return all_t, all_o, all_s, all_n, req.astype(np.int32)


def oracle_matches(all_t, all_o, all_s, all_n, req, ns, stride, greedy):
    idx = om.BlendIndex(C)
    for t, o, s, n in zip(all_t, all_o, all_s, all_n):
        idx.add(t.tolist(), int(o), int(s), int(n))
    m = idx.match(req.tolist(), ns, stride)
    return om.leftmost_greedy(m, C) if greedy else m


@pytest.mark.parametrize("ns,stride,greedy", [(1, 1, True), (2, 1, True), (1, 1, False), (2, 2, False), (1, 4, True)])
def test_matcher_equals_oracle(cb, ns, stride, greedy):
    all_t, all_o, all_s, all_n, req = build_case()
    index = cb.FragmentIndex(C, all_t, all_o, all_s, all_n, max_tokens=len(req))
    got = index.match(torch.from_numpy(req).cuda(), ns, stride, greedy)
    want = oracle_matches(all_t, all_o, all_s, all_n, req, ns, stride, greedy)
    assert len(want) > (10 if stride == 1 else 3)
    assert got == [tuple(int(v) for v in w) for w in want]
    index.close()


def test_matcher_edges(cb):
    all_t, all_o, all_s, all_n, req = build_case(seed=8, n_chunks=50, n_tokens=4096)
    index = cb.FragmentIndex(C, all_t, all_o, all_s, all_n, max_tokens=4096)
    assert index.size(3) == C and index.size(2) <= len(all_o)
    t = torch.from_numpy(req).cuda()
    assert index.match(t[:C - 1], 1) == []                 # shorter than a chunk: nothing to probe
    assert index.match(t[:0], 1) == []
    full = index.match(t, 1, greedy=False)
    part = index.match(t, 1, greedy=False, max_out=2)       # only the first max_out are written
    assert part == full[:2]
    with pytest.raises(cb.CacheBlendError):
        index.match(torch.zeros(5000, dtype=torch.int32, device="cuda"), 1)   # beyond max_tokens
    empty = cb.FragmentIndex(C, np.zeros((0, C), np.uint32), [], [], [], max_tokens=4096)
    assert empty.match(t, 1) == []
    index.close()
    empty.close()


@pytest.mark.parametrize("stride,greedy", [(1, True), (1, False), (3, True)])
def test_matcher_low_entropy_request(cb, stride, greedy):
    """A low-entropy request: a run of one repeated token, where every window verifies against the indexed
    chunk of that token (thousands of verified windows of one content).  Its occupants (three in the
    requester's namespace, one in another) are taken in position order and leftmost-greedy keeps windows
    a chunk apart; two more contents of mixed tokens are planted after the run."""
    n_tokens = 12288
    run = np.full((1, C), 77, np.uint32)
    mixed = np.stack([workload.tokens(3, 500 + i, C, VOCAB) for i in range(2)]).astype(np.uint32)
    all_t = np.concatenate([run, run, run, run, mixed])        # the run's content under four occupants
    all_o = np.array([1, 2, 3, 4, 5, 6], np.int32)
    all_s = np.array([0, 512, 1024, 0, 256, 768], np.int32)
    all_n = np.array([1, 1, 1, 2, 1, 1], np.int32)
    req = np.full(n_tokens, 77, np.int32)
    req[9000:9000 + C] = mixed[0]
    req[9400:9400 + C] = mixed[1]
    index = cb.FragmentIndex(C, all_t, all_o, all_s, all_n, max_tokens=n_tokens)
    got = index.match(torch.from_numpy(req).cuda(), 1, stride, greedy)
    want = oracle_matches(all_t, all_o, all_s, all_n, req, 1, stride, greedy)
    assert len(want) >= 2
    assert got == [tuple(int(v) for v in w) for w in want]
    index.close()
