"""The layer-oracle pins are sensitive: plant plausible mistakes in a copy of
oracle/layer.py (on the CPU) and check that the pins reject every one."""
import importlib.util
import os

import pytest

import oracle.layer as layer_mod

from . import test_layer_oracle as pins

SRC = layer_mod.__file__

MUTATIONS = {
    # taps applied in the wrong order (tap 0 on the current token)
    "reversed_taps": ("out += w[:, i] * xp[:, i:i + T, :]", "out += w[:, K - 1 - i] * xp[:, i:i + T, :]"),
    # the carried state dropped
    "state_ignored": ("prev = np.zeros((B, K - 1, C)) if state is None else f64(state)", "prev = np.zeros((B, K - 1, C))"),
    # state out taken from the wrong end
    "state_from_front": ("return out, xp[:, T:, :].copy()", "return out, xp[:, :K - 1, :].copy()"),
    # SiLU with the wrong sign inside the sigmoid
    "silu_sign": ("return u / (1.0 + np.exp(-u))", "return u / (1.0 + np.exp(u))"),
    # softplus replaced by exp
    "softplus_exp": ("alpha = np.exp(-np.exp(A) * softplus(a_raw + b_alpha))", "alpha = np.exp(-np.exp(A) * np.exp(a_raw + b_alpha))"),
    # exp(A) dropped from the decay exponent
    "A_dropped": ("alpha = np.exp(-np.exp(A) * softplus(a_raw + b_alpha))", "alpha = np.exp(-softplus(a_raw + b_alpha))"),
    # plain RMSNorm weight instead of zero-centred (1 + w)
    "weight_not_zero_centred": ("* (1.0 + w)", "* w"),
    # RMS over the whole tensor instead of per row
    "rms_wrong_axis": ("np.mean(y * y, axis=-1, keepdims=True)", "np.mean(y * y)"),
    # L2 norm over the whole tensor instead of per row
    "l2_wrong_axis": ("np.sum(u * u, axis=-1, keepdims=True)", "np.sum(u * u)"),
    # output gate applied as SiLU instead of sigmoid
    "silu_gate": ("return sigmoid(z) * rmsnorm_zc(y, w_norm, eps)", "return silu(z) * rmsnorm_zc(y, w_norm, eps)"),
    # the prologue's wiring: v normalised like q and k
    "v_normalised": ("v, sv = feature(xv, wv, state_v, False)", "v, sv = feature(xv, wv, state_v, True)"),
    # the incoming convolution states of q and k swapped
    "qk_states_swapped": ("q, sq = feature(xq, wq, state_q, True)\n    k, sk = feature(xk, wk, state_k, True)",
                          "q, sq = feature(xq, wq, state_k, True)\n    k, sk = feature(xk, wk, state_q, True)"),
    # q convolved with k's taps
    "q_reads_k_taps": ("q, sq = feature(xq, wq, state_q, True)", "q, sq = feature(xq, wk, state_q, True)"),
    # the decay and write gates fed each other's pre-activations
    "gate_inputs_swapped": ("alpha, beta = gates(a_raw, b_raw, A, b_alpha)", "alpha, beta = gates(b_raw, a_raw, A, b_alpha)"),
    # the outgoing states of q and k returned under each other's names
    "qk_states_out_swapped": ("state_q=sq, state_k=sk", "state_q=sk, state_k=sq"),
}

PIN_TESTS = [
    pins.test_conv_current_tap_is_identity_and_first_tap_is_a_shift,
    pins.test_conv_impulse_response_is_the_reversed_taps,
    pins.test_conv_state_carries_across_a_split,
    pins.test_conv_brute_force_small,
    pins.test_silu_closed_forms,
    pins.test_sigmoid_and_softplus_closed_forms,
    pins.test_gates_closed_forms,
    pins.test_l2norm_unit_rows_scale_invariance,
    pins.test_rmsnorm_zero_centred_closed_forms,
    pins.test_epilogue_gate_limits,
    pins.test_prologue_features_brute_force_tiny,
    pins.test_prologue_whole_brute_force_tiny,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_layer_pins_reject_mutation(name, tmp_path, monkeypatch):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert before in src, f"mutation anchor for {name} not found"
    path = tmp_path / "layer_mut.py"
    path.write_text(src.replace(before, after))
    spec = importlib.util.spec_from_file_location("layer_mut", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(pins, "L", mod)
    caught = 0
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin rejects mutation {name}"
