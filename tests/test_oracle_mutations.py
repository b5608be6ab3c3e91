"""The oracle's pins are tight: each plausible mistake, planted in the oracle
on the CPU (monkeypatch, undone after the test), makes at least one pin of
tests/test_oracle_pins.py fail.  A mutation that every pin let through would
mean a mistake of that kind could hide in the oracle."""

import numpy as np
import pytest

from oracle import costmodel, numerics, partition, sample, topology
from tests import test_oracle_pins as pins


def _caught(checks):
    """True when at least one check raises AssertionError."""
    for check in checks:
        try:
            check()
        except AssertionError:
            return True
    return False


def test_btree_children_swapped(monkeypatch, golden):
    orig = topology.btree

    def btree(n, r):
        u, d0, d1, t = orig(n, r)
        return u, d1, d0, t
    monkeypatch.setattr(topology, "btree", btree)
    assert _caught([lambda: pins.test_dtree4_figure(golden), pins.test_hand_derived_trees_r8_r7])


def test_btree_parent_type_inverted(monkeypatch):
    orig = topology.btree

    def btree(n, r):
        u, d0, d1, t = orig(n, r)
        return u, d0, d1, (1 - t if t in (0, 1) else t)
    monkeypatch.setattr(topology, "btree", btree)
    assert _caught([pins.test_btree_root_and_parent_types, pins.test_split_tree_two_by_two_by_hand])


def test_odd_node_count_mirrored_instead_of_shifted(monkeypatch, golden):
    btree = topology.btree

    def dtree(n, r):
        u, a, b, t = btree(n, n - 1 - r)
        back = lambda x: -1 if x == -1 else n - 1 - x  # noqa: E731
        return btree(n, r), (back(u), back(a), back(b), t)
    monkeypatch.setattr(topology, "dtree", dtree)
    assert _caught([lambda: pins.test_probe_table(golden),
                    lambda: pins.test_odd_overlap_at_node0(5)])


def test_children_prepended_to_down(monkeypatch, golden):
    def set_down(t, child):
        if child != -1:
            t.down = [child] + t.down[:2]
    monkeypatch.setattr(topology, "_set_down", set_down)
    assert _caught([lambda: pins.test_dtree4_figure(golden),
                    pins.test_tree_local_first_then_children_in_slot_order,
                    pins.test_hand_derived_trees_r8_r7])


def test_bf16_narrowing_truncates(monkeypatch):
    def f32_to_bf16_bits(x):
        b = np.asarray(x, dtype=np.float32).view(np.uint32)
        return (b >> 16).astype(np.uint16)
    monkeypatch.setattr(numerics, "f32_to_bf16_bits", f32_to_bf16_bits)
    assert _caught([pins.test_bf16_rne_matches_torch])


def test_max_ignores_signed_zero(monkeypatch):
    def combine(op, acc, other):
        acc = np.asarray(acc, dtype=np.float32)
        other = np.asarray(other, dtype=np.float32)
        if op == numerics.SUM:
            return np.add(acc, other, dtype=np.float32)
        return np.maximum(acc, other).astype(np.float32)
    monkeypatch.setattr(numerics, "combine", combine)
    assert _caught([pins.test_max_total_order_on_signed_zero])


def test_sum_accumulates_in_fp64(monkeypatch):
    def combine(op, acc, other):
        acc = np.asarray(acc, dtype=np.float64)
        other = np.asarray(other, dtype=np.float64)
        if op == numerics.SUM:
            return acc + other
        take = (other > acc) | ((other == acc) & np.signbit(acc) & ~np.signbit(other))
        return np.where(take, other, acc)
    monkeypatch.setattr(numerics, "combine", combine)
    assert _caught([pins.test_chain_fold_order, pins.test_ring_fold_starts_at_block_owner,
                    pins.test_tree_local_first_then_children_in_slot_order])


def test_block_remainder_at_the_end(monkeypatch):
    def split_sizes(total, parts):
        q, m = divmod(total, parts)
        return [q + (1 if i >= parts - m else 0) for i in range(parts)]
    monkeypatch.setattr(partition, "split_sizes", split_sizes)
    assert _caught([pins.test_partition_covers_message])


def test_ring_fold_starts_one_rank_late(monkeypatch):
    orig = sample.ring_fold_start

    def ring_fold_start(e, count, elem_size, R, n_channels, chunk_elems):
        return (orig(e, count, elem_size, R, n_channels, chunk_elems) + 1) % R
    monkeypatch.setattr(sample, "ring_fold_start", ring_fold_start)
    assert _caught([lambda: pins.test_sampler_matches_literal_simulation(pins.RING)])


def test_ring_stage_count_off_by_two(monkeypatch):
    def ring_terms(N, M):
        return 2 * N, 2.0 * (N - 1) / N * M
    monkeypatch.setattr(costmodel, "ring_terms", ring_terms)
    assert _caught([pins.test_cost_model_step_counts_and_traffic])


def test_tree_traffic_halved(monkeypatch):
    def tree_terms(D, M):
        return 2 * D, 1.0 * M
    monkeypatch.setattr(costmodel, "tree_terms", tree_terms)
    assert _caught([pins.test_cost_model_step_counts_and_traffic])


@pytest.mark.parametrize("name", ["test_btree_root_and_parent_types", "test_partition_covers_message",
                                  "test_max_total_order_on_signed_zero"])
def test_pins_pass_unmutated(name):
    """The same pins pass on the oracle as written (so a caught mutation is
    the mutation's doing)."""
    getattr(pins, name)()
