"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import oracle
import pins


def test_bookkeeping_worked_example():
    pins.check_bookkeeping(oracle.default())


def test_route_io_worked_example():
    pins.check_route_io(oracle.default())


def test_scalar_end_to_end_worked_example():
    pins.check_scalar_e2e(oracle.default())


def test_shared_expert_worked_example():
    pins.check_shared(oracle.default())


def test_shape_trace():
    pins.check_shape_trace(oracle.default())


def test_brute_force_all_experts_masked():
    pins.check_brute_force(oracle.default())


def test_closed_forms_and_special_cases():
    pins.check_closed_forms(oracle.default())


def test_ties_go_to_lower_expert_index():
    pins.check_ties(oracle.default())


def test_grouping_matches_numpy_stable_sort():
    pins.check_align_vs_numpy(oracle.default())


def test_batch_invariance():
    pins.check_batch_invariance(oracle.default())


def test_pitfall_variants_are_rejected_by_the_pins():
    """The printed numbers tell the correct method from the pitfalls listed
    in the M03 drill ("common mistakes"): repeat instead of repeat_interleave,
    assignment instead of accumulation, top-k logits then softmax."""
    import numpy as np
    g = pins.golden()
    b = g["bookkeeping"]
    wrong_tok = np.tile(np.arange(b["N"]), b["k"])          # arange(N).repeat(k)
    assert wrong_tok.tolist() == b["flat_tok_wrong_repeat"] != b["flat_tok"]
    s = g["scalar_e2e"]
    # assignment: token 0 keeps only the last expert written (expert 1)
    assigned = s["weights"][0][1] * s["expert_out"][0][1]
    assert abs(assigned - s["out_if_assigned_token0"]) < 1e-4
    assert abs(assigned - s["out"][0][0]) > 1.0
    r = g["route_io"]
    import scipy.special
    x = np.array(r["x"])
    top_first = scipy.special.softmax(np.sort(x, axis=1)[:, ::-1][:, :2], axis=1)
    # equals the renormalised weights, but not the raw ones
    assert np.allclose(top_first, r["weights_norm"], atol=1e-4)
    assert not np.allclose(top_first, r["weights_raw"], atol=1e-2)


def test_fused_add_rmsnorm():
    pins.check_add_rmsnorm(oracle.default())
