"""The seeded generator: determinism, layout, canaries, bf16 rounding."""

import numpy as np
import pytest

from speculative_decoding_verification_47_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 10,
                        [0.0, -0.0, 1e-40, 3.0e38, np.inf, -np.inf]])
    ours = wl.f64_to_bf16_bits(x)
    ref = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    np.testing.assert_array_equal(ours.view(np.int16), ref.numpy())


def test_deterministic_and_shapes():
    a = wl.synth_verify("t", 3, 4, 257, wl.BF16, [4, 2, 0], [1.0, 0.7, 0.1],
                        [0.5, 1.0, 2.0], [0, 1, 0], top_p=0.9)
    b = wl.synth_verify("t", 3, 4, 257, wl.BF16, [4, 2, 0], [1.0, 0.7, 0.1],
                        [0.5, 1.0, 2.0], [0, 1, 0], top_p=0.9, threads=4)
    for f in ("target", "draft", "draft_tokens", "uniforms"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert a.target.shape == (3, 5, 257) and a.draft.shape == (3, 4, 257)
    assert a.target.dtype == np.uint16


def test_canaries_in_padding():
    a = wl.synth_verify("t", 2, 5, 64, wl.F32, [2, 5], 1.0, 0.5, 0)
    assert np.isnan(a.target[0, 3:]).all() and not np.isnan(a.target[0, :3]).any()
    assert np.isnan(a.draft[0, 2:]).all() and not np.isnan(a.draft[0, :2]).any()
    assert (a.draft_tokens[0, 2:] == -1).all() and (a.draft_tokens[0, :2] >= 0).all()
    assert np.isnan(a.uniforms[0, 2:5]).all() and not np.isnan(a.uniforms[0, 5])
    u = a.uniforms[1]
    assert ((u >= 0) & (u < 1)).all()
    assert np.all(u * 2**24 == np.round(u * 2**24))


def test_greedy_rows_draft_argmax():
    a = wl.synth_verify("t", 2, 3, 100, wl.BF16, 3, 0.7, 1.0, [1, 1])
    z = wl.bf16_bits_to_f32(a.draft)
    for b in range(2):
        for i in range(3):
            assert a.draft_tokens[b, i] == int(np.argmax(z[b, i]))


def test_c0_rounds_equal_batched():
    full = wl.config_c0_batched(rounds=4, V=500)
    for r in range(4):
        one = wl.config_c0(r, V=500)
        np.testing.assert_array_equal(one.target[0], full.target[r])
        np.testing.assert_array_equal(one.draft_tokens[0], full.draft_tokens[r])


def test_c2_row_params():
    k, T, s = wl.c2_row_params(256)
    assert k.min() >= 2 and k.max() <= 8
    assert set(np.unique(T).tolist()) <= {np.float32(0.1), np.float32(0.7), np.float32(1.0)}
    assert set(np.unique(s).tolist()) <= {0.3, 1.0, 2.0}


def test_row_spec_regenerates_the_batch_sequences():
    """bench.py's CPU legs regenerate single sequences from the row spec; they
    must be the sequences of the batch workload."""
    for name, B in (("c1", 5), ("c2", 6), ("c3", 4)):
        spec = wl.row_spec(name, B)
        w = wl.config_by_name(name, B)
        assert (spec.B, spec.K, spec.V, spec.dtype, spec.top_p) == (w.B, w.K, w.V, w.dtype, w.top_p)
        np.testing.assert_array_equal(spec.mode, w.mode)
        np.testing.assert_array_equal(spec.k_per_row, w.k_per_row)
        for b in (0, B - 1):
            t, d, x, u = spec.sequence(b)
            np.testing.assert_array_equal(t, w.target[b])
            np.testing.assert_array_equal(d, w.draft[b])
            np.testing.assert_array_equal(x, w.draft_tokens[b])
            np.testing.assert_array_equal(u, w.uniforms[b])


def test_paged_round_tables_cover_each_sequence_exactly():
    r = wl.paged_round(B=64, max_pages=32, page_size=16, seed=7)
    ids = r.block_table[r.block_table >= 0]
    assert len(np.unique(ids)) == len(ids) and ids.max() < r.pool_pages
    for b in range(64):
        need = -(-(int(r.seq_lens[b]) + int(r.k_per_row[b])) // 16)
        assert np.all(r.block_table[b, :need] >= 0) and np.all(r.block_table[b, need:] == -1)
        assert 0 <= r.n_accepted[b] <= r.k_per_row[b] and 2 <= r.k_per_row[b] <= 8


def test_dynk_history_ranges():
    n, k = wl.dynk_history(B=32, rounds=100, seed=3)
    assert n.shape == k.shape == (100, 32) and n.dtype == k.dtype == np.int32
    assert k.min() >= 2 and k.max() <= 8 and n.min() >= 0 and np.all(n <= k)
    assert len(np.unique(n)) == 9  # every count 0..8 occurs
