"""The seeded input module: length mixes and determinism (no GPU)."""
import chain_synth as cs


def test_varlen_lengths_cover_total_within_bounds():
    for seed in (0, 7, 8):
        lens = cs.varlen_lengths(131072, 1024, 16384, seed)
        assert sum(lens) == 131072
        assert all(1024 <= L <= 16384 for L in lens[:-1])
        assert 1 <= lens[-1] <= 16384


def test_varlen_lengths_are_seeded():
    assert cs.varlen_lengths(50000, 100, 5000, 3) == cs.varlen_lengths(50000, 100, 5000, 3)
    assert cs.varlen_lengths(50000, 100, 5000, 3) != cs.varlen_lengths(50000, 100, 5000, 4)


def test_workload_seeds_are_distinct():
    seeds = [w.seed for w in cs.WORKLOADS.values()]
    assert len(seeds) == len(set(seeds))
