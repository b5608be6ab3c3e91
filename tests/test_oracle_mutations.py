"""The oracle's pins are tight: each plausible mistake, planted in the oracle
on the CPU (monkeypatch, undone after the test), makes at least one pin of
tests/test_oracle_pins.py fail.  A mutation that every pin let through would
mean a mistake of that kind could hide in the oracle."""

import functools
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from oracle import api, costmodel, numerics, partition, sample, schedules, topology
from tests import test_oracle_pins as pins


def _caught(checks):
    """True when at least one check fails: an assertion, or an error raised
    by the mutated oracle (a tree that no longer reaches every rank, an index
    out of range)."""
    for check in checks:
        try:
            check()
        except Exception:
            return True
    return False


def _rewrite(monkeypatch, module, name, old, new):
    """Install, for the test's duration, module.name with the one occurrence
    of ``old`` in its source replaced by ``new``."""
    for attr, fn in list(vars(module).items()):
        if hasattr(fn, "cache_clear"):
            # a cache of the test's own, so that nothing computed under the
            # mutation outlives it (or was computed before it)
            monkeypatch.setattr(module, attr, functools.lru_cache(maxsize=None)(fn.__wrapped__))
    src = textwrap.dedent(inspect.getsource(getattr(module, name)))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(module))
    exec(compile(src.replace(old, new), module.__file__, "exec"), ns)
    if getattr(oracle, name, None) is getattr(module, name):   # re-exported by the package
        monkeypatch.setattr(oracle, name, ns[name])
    monkeypatch.setattr(module, name, ns[name])


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


# ------------------------------------------ one expression of the oracle changed
# (module, function, original text, mutated text, the pins expected to catch it)
REWRITES = [
    ("ring sends to the left neighbour", schedules, "ring_allreduce_loop",
     "dst = (r + 1) % R", "dst = (r - 1) % R",
     ["test_ring_trace_figure1"]),
    ("ring all-gather forwards the block one step early", schedules, "ring_allreduce_loop",
     "(r + 1 - s) % R, held[r][(r + 1 - s) % R]", "(r - s) % R, held[r][(r - s) % R]",
     ["test_ring_trace_figure1", "test_brute_force_exact_small_integers"]),
    ("ReduceScatter uses the AllReduce block labels", schedules, "ring_reduce_scatter",
     "(r - s - 1) % R, held[r][(r - s - 1) % R]", "(r - s) % R, held[r][(r - s) % R]",
     ["test_reduce_scatter_blocks_and_order", "test_each_rank_contributes_once"]),
    ("AllGather forwards the block it received last step", schedules, "ring_allgather",
     "(r - s) % R, held[r][(r - s) % R]", "(r - s + 1) % R, held[r][(r - s + 1) % R]",
     ["test_allgather_is_concatenation"]),
    ("tree reduce leaves out the local input", schedules, "tree_allreduce_chunk",
     "acc = xs[v][start:start + length].copy()", "acc = np.zeros(length, np.float32)",
     ["test_each_rank_contributes_once", "test_two_rank_example"]),
    ("tree broadcast forwards the child's own partial", schedules, "tree_allreduce_chunk",
     "result[c] = result[v].copy()", "result[c] = partial[c].copy()",
     ["test_each_rank_contributes_once", "test_brute_force_exact_small_integers"]),
    ("tree folds children in reverse slot order", schedules, "tree_allreduce_chunk",
     "for c in tree[v].down:\n                if c != -1:\n                    acc",
     "for c in reversed(tree[v].down):\n                if c != -1:\n                    acc",
     ["test_tree_local_first_then_children_in_slot_order"]),
    ("first tree takes the smaller half of the channels", topology, "channel_tree_index",
     "(n_channels + 1) // 2", "n_channels // 2",
     ["test_channel_to_tree_split"]),
    ("tree halves swapped", topology, "channel_tree_index",
     "return 0 if channel", "return 1 if channel",
     ["test_channel_to_tree_split"]),
    ("parent is the farther of the higher-level neighbours", topology, "_parents",
     "_level(left) < _level(right)", "_level(left) > _level(right)",
     ["test_dtree4_figure", "test_hand_derived_trees_r8_r7", "test_tree_invariants"]),
    ("parent on the right even past the end", topology, "_parents",
     "if right is None or", "if right is not None and",
     ["test_dtree4_figure", "test_hand_derived_trees_r8_r7", "test_tree_invariants"]),
    ("level from the highest set bit", topology, "_level",
     "v & -v", "1 << (v.bit_length() - 1)",
     ["test_dtree4_figure", "test_hand_derived_trees_r8_r7", "test_tree_invariants"]),
    ("root not above every level", topology, "_level",
     "math.inf if v == 0", "0 if v == 0",
     ["test_btree_root_and_parent_types"]),
    ("odd double tree shifted the other way", topology, "dtree",
     "btree(n, (r - 1 + n) % n)", "btree(n, (r + 1) % n)",
     ["test_probe_table", "test_odd_overlap_at_node0", "test_tree_invariants"]),
    ("parent head hangs under the other child head", topology, "build_dtree",
     "(ttc0 if ptype == 0 else ttc1)[u]", "(ttc1 if ptype == 0 else ttc0)[u]",
     ["test_split_tree_two_by_two_by_hand", "test_balanced_tree_four_by_two_by_hand"]),
    ("second child node attached to the child0 head", topology, "build_dtree",
     "_set_down(per_rank[ttc1[k]], ttp[d1])", "_set_down(per_rank[ttc0[k]], ttp[d1])",
     ["test_balanced_tree_four_by_two_by_hand"]),
    ("intra order ignored", topology, "build_dtree",
     "k * L + order[i]", "k * L + i",
     ["test_active_trees_table"]),
    ("SPLIT_TREE with the BALANCED_TREE heads", topology, "head_indices",
     "return 0, 1, 1", "return 0, 1, 0",
     ["test_split_tree_two_by_two_by_hand"]),
    ("BALANCED_TREE with its child heads swapped", topology, "head_indices",
     "return 0, 1, 0", "return 0, 0, 1",
     ["test_balanced_tree_four_by_two_by_hand"]),
    ("per-hop rounding left out", api, "allreduce",
     "hop = lambda x: numerics.to_f32(numerics.from_f32(x, dtype), dtype)", "hop = lambda x: x",
     ["test_hop_rounding_bf16_by_hand"]),
    ("bf16 widened with a 15-bit shift", numerics, "bf16_bits_to_f32",
     "<< np.uint32(16)", "<< np.uint32(15)",
     ["test_bf16_rne_matches_torch"]),
    ("tree depth counted in nodes, not edges", topology, "exact_depth",
     "worst = max(worst, d)", "worst = max(worst, d + 1)",
     ["test_probe_table"]),
    ("internal nodes leave out the root", topology, "internal_nodes",
     "if any(c != -1 for c in t.down)", "if t.up != -1 and any(c != -1 for c in t.down)",
     ["test_probe_table", "test_odd_overlap_at_node0"]),
    ("ring prev points forward", topology, "build_ring",
     "(r - 1 + R) % R", "(r + 1) % R",
     ["test_ring_topology"]),
    ("ring all-gather sends not counted", schedules, "ring_allreduce_loop",
     "held[(r + 1) % R][j] = msg\n            if counters is not None:\n"
     "                counters.sent[r] += msg.size",
     "held[(r + 1) % R][j] = msg\n            if counters is not None:\n"
     "                counters.sent[r] += 0",
     ["test_ring_traffic_closed_form", "test_ring_four_ranks_sends_one_and_a_half_S"]),
    ("tree broadcast sends not counted", schedules, "tree_allreduce_chunk",
     "nxt.append(c)\n                    if counters is not None:\n"
     "                        counters.sent[v] += length",
     "nxt.append(c)\n                    if counters is not None:\n"
     "                        counters.sent[v] += 0",
     ["test_tree_sends_at_most_2S_per_rank_even_mirror"]),
    ("log2 rounded up", topology, "log2i",
     "n >>= 1", "n = (n + 1) >> 1",
     ["test_log2i_is_floor"]),
    ("tree log line with up and rank swapped", topology, "format_tree_log",
     "(channel, t.up, r, kids)", "(channel, r, t.up, kids)",
     ["test_active_chains_and_log_line"]),
    ("prediction divides by the inverse bandwidth", costmodel, "predict",
     "traffic * inv_bw", "traffic / inv_bw",
     ["test_cost_model_selects_lower_prediction_by_hand", "test_cost_model_fit_recovers_parameters"]),
    ("narrowing uses the other 16-bit format", numerics, "from_f32",
     "return f32_to_f16_bits(x)", "return f32_to_bf16_bits(x)",
     ["test_within_fp64_bounds"]),
    ("ReduceScatter sampler starts at the owner", sample, "reduce_scatter_element",
     "(block + 1 + k) % R", "(block + k) % R",
     ["test_reduce_scatter_sampler_matches_literal"]),
    ("ring loop of one chunk instead of R", partition, "ring_blocks",
     "step = R * chunk_elems", "step = chunk_elems",
     ["test_partition_small_ring_case"]),
    ("channels split in elements, not 16-byte grains", partition, "channel_ranges",
     "grains = -(-count // U)", "grains, U = count, 1",
     ["test_partition_covers_message"]),
    ("fp16 narrowing rounds ties away from zero", numerics, "f32_to_f16_bits",
     "(rem > half) | ((rem == half) & ((q & 1) == 1))", "rem >= half",
     ["test_f16_rne_matches_numpy_and_torch"]),
    ("fp16 narrowing ignores the subnormal range", numerics, "f32_to_f16_bits",
     "d = np.maximum(13, 126 - e_eff)", "d = np.full_like(e_eff, 13)",
     ["test_f16_rne_matches_numpy_and_torch"]),
    ("fp16 widening with exponent bias 16", numerics, "f16_bits_to_f32",
     "(np.maximum(e, 1) - 25)", "(np.maximum(e, 1) - 26)",
     ["test_f16_rne_matches_numpy_and_torch"]),
    ("fp64 sum accumulated in fp32", api, "fp64_sum",
     "acc += x.astype(np.float64)", "acc = (acc.astype(np.float32) + x).astype(np.float64)",
     ["test_fp64_sum_exact_where_fp64_is"]),
    ("fp64 max starts from zero", api, "fp64_max",
     "-np.inf", "0.0",
     ["test_brute_force_exact_small_integers", "test_fp64_sum_exact_where_fp64_is"]),
    ("sampler: element at a channel's end counted in the channel", sample, "channel_of",
     "cs <= e < cs + cn", "cs < e <= cs + cn",
     ["test_sampler_matches_literal_simulation"]),
    ("sampler: tree children folded in reverse", sample, "tree_fold",
     "for c in tree[v].down:", "for c in reversed(tree[v].down):",
     ["test_sampler_matches_literal_simulation"]),
    ("crossover of the wrong sign", costmodel, "crossover",
     "m = num / den", "m = -num / den",
     ["test_cost_model_crossover_matches_search"]),
    ("least-squares columns transposed", costmodel, "fit",
     "np.asarray(stages, float), np.asarray(traffic, float)",
     "np.asarray(traffic, float), np.asarray(stages, float)",
     ["test_cost_model_fit_recovers_parameters"]),
    ("relative fit without the weighting (absolute least squares)", costmodel, "fit_relative",
     "], float) / t,", "], float) / 1.0,",
     ["test_cost_model_relative_fit_by_hand"]),
    ("relative fit keeps samples whose time is not positive", costmodel, "fit_relative",
     "if t > 0]", "if t > 0 or t <= 0]",
     ["test_cost_model_relative_fit_by_hand"]),
    ("selection picks the slower algorithm", costmodel, "select",
     "t_ring(N, M, *ring) <= t_tree(D, M, *tree)", "t_ring(N, M, *ring) > t_tree(D, M, *tree)",
     ["test_cost_model_selects_lower_prediction_by_hand"]),
    ("tree cost model counts one pass of the tree", costmodel, "tree_terms",
     "return 2 * D, 2.0 * M", "return D, 2.0 * M",
     ["test_cost_model_step_counts_and_traffic"]),
]


def _pin_checks(names, golden):
    """The named pins as zero-argument checks, over every parameter value of
    their own ``parametrize`` marks (the golden fixture passed in)."""
    import itertools
    checks = []
    for name in names:
        fn = getattr(pins, name)
        grid = {"golden": [golden]}
        for mark in getattr(fn, "pytestmark", []):
            if mark.name == "parametrize":
                grid[mark.args[0]] = list(mark.args[1])
        params = list(inspect.signature(fn).parameters)
        for combo in itertools.product(*[grid[p] for p in params]):
            checks.append(lambda fn=fn, kw=dict(zip(params, combo)): fn(**kw))
    return checks


@pytest.mark.parametrize("what,module,name,old,new,catchers", REWRITES,
                         ids=[r[0] for r in REWRITES])
def test_rewrite_is_caught(monkeypatch, golden, what, module, name, old, new, catchers):
    _rewrite(monkeypatch, module, name, old, new)
    assert _caught(_pin_checks(catchers, golden)), what


@pytest.mark.parametrize("what,module,name,old,new,catchers", REWRITES,
                         ids=[r[0] for r in REWRITES])
def test_unchanged_rewrite_keeps_pins_green(monkeypatch, golden, what, module, name, old, new,
                                            catchers):
    """The rewrite machinery itself (recompiling the function from its source
    in a copy of its module's namespace) changes nothing: with the text put
    back unchanged, the same pins pass."""
    _rewrite(monkeypatch, module, name, old, old)
    for check in _pin_checks(catchers, golden):
        check()


@pytest.mark.parametrize("name", ["test_btree_root_and_parent_types", "test_partition_covers_message",
                                  "test_max_total_order_on_signed_zero"])
def test_pins_pass_unmutated(name):
    """The same pins pass on the oracle as written (so a caught mutation is
    the mutation's doing)."""
    getattr(pins, name)()
