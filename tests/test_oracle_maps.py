"""Pins for the oracle's sparse rearrange and index maps (CPU only).

The rearrange is "Open-Sora Plan" docs, section "Skiparse Attention", Single
Skip and Group Skip Implementation listings. Pins used here:
  * the einops library applied to the listings' own patterns;
  * the hand-derived golden fixture tests/golden/skiparse_scopes.txt (prose);
  * reverse o rearrange == identity, bijection, scope sizes;
  * the closed forms scope = i mod k / (i div k) mod k written out below.
"""
import os

import einops
import numpy as np
import pytest

from oracle import skiparse_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "skiparse_scopes.txt")
MODES = [(O.SINGLE, "single"), (O.GROUP, "group")]


def _shapes(mode):
    for k in (1, 2, 3, 4, 8):
        for mult in (1, 2, 5):
            N = mult * (k if mode == O.SINGLE else k * k) * 2
            for B in (1, 3):
                yield B, N, k


@pytest.mark.parametrize("mode,name", MODES)
def test_rearrange_matches_einops_patterns(mode, name):
    rng = np.random.default_rng(7)
    for B, N, k in _shapes(mode):
        x = rng.standard_normal((B, N, 5))
        if mode == O.SINGLE:
            ref = einops.rearrange(x, "b (g k) d -> (k b) g d", k=k)
            back = einops.rearrange(ref, "(k b) g d -> b (g k) d", k=k)
        else:
            ref = einops.rearrange(x, "b (n m k) d -> (m b) (n k) d", m=k, k=k)
            back = einops.rearrange(ref, "(m b) (n k) d -> b (n m k) d", m=k, k=k)
        got = O.rearrange(x, k, mode)
        assert np.array_equal(got, ref)
        assert np.array_equal(O.reverse(ref, k, mode), back)


@pytest.mark.parametrize("mode,name", MODES)
def test_reverse_of_rearrange_is_identity(mode, name):
    for B, N, k in _shapes(mode):
        x = np.arange(B * N * 3, dtype=np.int64).reshape(B, N, 3)
        assert np.array_equal(O.reverse(O.rearrange(x, k, mode), k, mode), x)


def test_golden_scopes_from_prose():
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, toks = line.split(":")
            mode_s, k, N, s = head.split()
            mode = O.SINGLE if mode_s == "single" else O.GROUP
            want = np.array([int(t) for t in toks.split()], dtype=np.int64)
            got = O.scope_tokens(int(N), int(k), mode, int(s))
            assert np.array_equal(got, want), line
            n += 1
    assert n >= 20


def _closed_form(N, k, mode):
    i = np.arange(N, dtype=np.int64)
    if mode == O.SINGLE:
        return i % k, i // k
    return (i // k) % k, (i // (k * k)) * k + i % k


@pytest.mark.parametrize("mode,name", MODES)
def test_index_maps_closed_form_and_bijection(mode, name):
    for k in (1, 2, 3, 4, 8):
        for N in (k * k * 4, k * k * 12, 4096 - 4096 % (k * k)):
            scope, pos = O.index_maps(N, k, mode)
            cs, cp = _closed_form(N, k, mode)
            assert np.array_equal(scope, cs) and np.array_equal(pos, cp)
            L = N // k
            # bijection onto k scopes x L positions, every scope exactly L tokens
            flat = scope * L + pos
            assert np.array_equal(np.sort(flat), np.arange(N))
            assert np.all(np.bincount(scope, minlength=k) == L)
            # inverse map back to the token id
            if mode == O.SINGLE:
                inv = pos * k + scope
            else:
                inv = (pos // k) * k * k + scope * k + pos % k
            assert np.array_equal(inv, np.arange(N))


@pytest.mark.parametrize("mode,name", MODES)
def test_scope_mates_match_prose_mask(mode, name):
    for k in (2, 3, 4):
        N = k * k * 6
        scope, _ = O.index_maps(N, k, mode)
        mask = O.skiparse_mask(N, k, mode)
        assert np.array_equal(scope[:, None] == scope[None, :], mask)
        i = np.arange(N)
        if mode == O.SINGLE:
            # every k-th token: j - i is a multiple of k
            assert np.array_equal(mask, ((i[:, None] - i[None, :]) % k) == 0)
        else:
            g = i // k
            assert np.array_equal(mask, ((g[:, None] - g[None, :]) % k) == 0)


def test_k1_is_identity():
    for mode, _ in MODES:
        x = np.random.default_rng(1).standard_normal((2, 12, 3))
        assert np.array_equal(O.rearrange(x, 1, mode), x)


@pytest.mark.parametrize("mode,name", MODES)
def test_prose_scopes_equal_the_rearrange_when_divisible(mode, name):
    """Where the listings' rearrange applies, the prose definition of a scope
    (the one used for every other N) gives exactly its rows."""
    for _, N, k in _shapes(mode):
        for s in range(k):
            ids = O.rearrange(np.arange(N, dtype=np.int64)[None, :], k, mode)[s]
            assert np.array_equal(O.prose_scope_tokens(N, k, mode, s), ids)


@pytest.mark.parametrize("mode,name", MODES)
def test_ragged_index_maps(mode, name):
    """Any N: the maps are a bijection of the tokens onto (scope, position < L_s),
    scope lengths differ by at most one token (single) or one group (group),
    lower scopes are never shorter, and the in-scope position inverts by the
    same closed forms as in the divisible case."""
    for k in (2, 3, 4, 5, 8):
        for N in range(1, 3 * k * k + 2):
            scope, pos = O.index_maps(N, k, mode)
            sizes = np.bincount(scope, minlength=k)
            assert sizes.sum() == N
            assert np.all(np.diff(sizes) <= 0)
            assert sizes[0] - sizes[-1] <= (1 if mode == O.SINGLE else k)
            flat = {(int(s_), int(p_)) for s_, p_ in zip(scope, pos)}
            assert len(flat) == N and all(p_ < sizes[s_] for s_, p_ in flat)
            if mode == O.SINGLE:
                inv = pos * k + scope
            else:
                inv = (pos // k) * k * k + scope * k + pos % k
            assert np.array_equal(inv, np.arange(N))
            mask = O.skiparse_mask(N, k, mode)
            assert np.array_equal(scope[:, None] == scope[None, :], mask)
