"""Plant plausible mistakes in the oracle (on the CPU, one at a time) and check
that the pins catch each one: evidence that the pins constrain every step."""
import numpy as np
import pytest

import oracle
from oracle import draft, philox, sampling, schedule, tv, verify
import tests.test_oracle_draft as T_draft
import tests.test_oracle_schedule as T_sched
import tests.test_oracle_tv as T_tv
import tests.test_oracle_verify as T_verify


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_gumbel_sign_slip_is_caught(monkeypatch):
    monkeypatch.setattr(philox, "gumbel", lambda u: np.log(-np.log(np.asarray(u, np.float64))))
    assert _fails(T_draft.test_gumbel_max_matches_softmax)


def test_one_word_per_philox_block_is_caught(monkeypatch):
    # the four indices of a Philox block sharing one word (word 0) instead of word v & 3
    orig = philox.row_words

    def bad(seed, b, k, stream, V):
        w = orig(seed, b, k, stream, -(-V // 4) * 4)
        return np.repeat(w[:, 0::4], 4, axis=1)[:, :V]
    monkeypatch.setattr(philox, "row_words", bad)
    assert _fails(T_draft.test_gumbel_max_matches_softmax)
    assert _fails(T_draft.test_gumbel_max_is_the_literal_definition)


def test_noise_keyed_without_the_request_is_caught(monkeypatch):
    # every request of a batch drawing the same noise (request index dropped from the counter)
    orig = philox.row_words
    monkeypatch.setattr(philox, "row_words", lambda seed, b, k, stream, V: orig(seed, np.zeros_like(b), k, stream, V))
    assert _fails(T_draft.test_gumbel_max_matches_softmax)
    assert _fails(T_draft.test_gumbel_max_noise_is_keyed_by_index_request_position_stream)


def test_verifier_token_on_the_draft_stream_is_caught(monkeypatch):
    # the residual drawn with the same noise that proposed x_k (stream 0 at (b, k)):
    # the residual draw is then tied to the rejected proposal and loses its law
    monkeypatch.setattr(philox, "STREAM_VERIFY_TOKEN", philox.STREAM_DRAFT_TOKEN)
    assert _fails(T_verify.test_token_after_a_rejection_follows_the_residual)


def test_transposed_bias_is_caught(monkeypatch):
    def bad(W1, W2, prev):
        E = np.asarray(W2, np.float64)[np.asarray(prev)]
        return E @ np.asarray(W1, np.float64).T
    monkeypatch.setattr(draft, "markov_bias", bad)
    assert _fails(T_draft.test_markov_bias_orientation)
    assert _fails(T_draft.test_chain_uses_previous_token)


def test_anchor_instead_of_previous_token_is_caught(monkeypatch):
    orig = draft.draft_block

    def bad(U, h, W1, W2, w, bias, x0, temperature, seed, forced_tokens=None):
        B, G, _ = np.shape(U)
        return orig(U, h, W1, W2, w, bias, x0, temperature, seed,
                    forced_tokens=np.repeat(np.asarray(x0)[:, None], G, axis=1))
    monkeypatch.setattr(draft, "draft_block", bad)
    assert _fails(T_draft.test_chain_uses_previous_token)
    assert _fails(T_draft.test_confidence_markov_part_reads_previous_token)


def test_theta_without_per_row_normalisation_is_caught(monkeypatch):
    from fractions import Fraction

    def bad(a, sps):
        a = np.asarray(a, np.float32)
        B, G = a.shape
        pairs = sorted(((b, j) for b in range(B) for j in range(1, G + 1)),
                       key=lambda p: (-float(a[p[0], p[1] - 1]), p[0], p[1]))
        ell, E, N = np.zeros(B, np.int64), Fraction(B), B
        best = float(E) * sps[N]
        for b, j in pairs:
            th = float(E + Fraction(float(a[b, j - 1]))) * sps[N + 1]
            if th > best:
                ell[b] += 1
                E += Fraction(float(a[b, j - 1]))
                N += 1
                best = th
            else:
                break
        return ell, N, best
    monkeypatch.setattr(schedule, "schedule_prefix", bad)
    assert _fails(T_sched.test_greedy_stop_is_global_optimum_for_rational_sps)


def test_non_strict_comparison_is_caught(monkeypatch):
    src = schedule.schedule_prefix

    def bad(a, sps):
        a = np.asarray(a, np.float32)
        eps_sps = np.asarray(sps, np.float64) * (1 + 1e-15)
        eps_sps[:a.shape[0] + 1] = np.asarray(sps)[:a.shape[0] + 1]
        return src(a, eps_sps)
    monkeypatch.setattr(schedule, "schedule_prefix", bad)
    assert _fails(T_sched.test_equal_theta_stops_the_scan)


def test_resampling_from_target_on_reject_is_caught(monkeypatch):
    # a classic slip: on a rejection draw from p_t instead of max(0, p_t - p_d)
    import oracle.verify as V
    monkeypatch.setattr(V, "draft_logits",
                        lambda U, W1, W2, x0, tokens, b, k, E=None: np.full((len(b), np.shape(U)[-1]), -np.inf))
    assert _fails(T_verify.test_first_emitted_token_follows_target)


def test_tv_missing_half_is_caught(monkeypatch):
    monkeypatch.setattr(tv, "accept_rate_tv",
                        lambda d, t: 1.0 - np.sum(np.abs(tv.softmax(d) - tv.softmax(t)), axis=-1))
    assert _fails(T_tv.test_disjoint_supports_give_zero)
    assert _fails(T_tv.test_two_point_closed_form)


def test_loss_ce_without_logsumexp_is_caught(monkeypatch):
    from oracle import loss as L
    import tests.test_oracle_loss as T_loss
    monkeypatch.setattr(L, "logsumexp_rows", lambda x: np.max(np.asarray(x, np.float64), axis=-1))
    assert _fails(T_loss.test_closed_forms)


def test_loss_bce_sign_slip_is_caught(monkeypatch):
    from oracle import loss as L
    import tests.test_oracle_loss as T_loss
    orig = L.softplus
    monkeypatch.setattr(L, "softplus", lambda s: orig(-np.asarray(s, np.float64)))
    assert _fails(T_loss.test_grad_s_matches_central_differences)


def test_loss_l1_gradient_without_the_softmax_mean_is_caught(monkeypatch):
    from oracle import loss as L
    import tests.test_oracle_loss as T_loss

    def bad_grad(d, t, target, conf_logit, omega, alpha_ce=L.ALPHA_CE, alpha_l1=L.ALPHA_L1, alpha_conf=L.ALPHA_CONF):
        p_d, p_t = L.softmax(d), L.softmax(t)
        g = np.asarray(omega, np.float64)[:, None] * alpha_l1 * 0.5 * p_d * np.sign(p_d - p_t)
        R = p_d.shape[0]
        oh = np.zeros_like(p_d)
        oh[np.arange(R), target] = 1.0
        g += np.asarray(omega, np.float64)[:, None] * alpha_ce * (p_d - oh)
        return g, np.zeros(R)
    monkeypatch.setattr(L, "dspark_loss_grad", bad_grad)
    assert _fails(T_loss.test_grad_d_matches_central_differences)


def test_rounds_sharing_one_key_is_caught(monkeypatch):
    from oracle import rounds as R
    import tests.test_oracle_rounds as T_rounds
    monkeypatch.setattr(R, "round_seed", lambda seed, i: int(seed))
    assert _fails(T_rounds.test_rounds_draw_with_their_own_keys)


def test_rounds_dropping_the_verifier_token_is_caught(monkeypatch):
    from oracle import rounds as R
    import tests.test_oracle_rounds as T_rounds

    def bad(x, n_accept, next_token):
        x = np.asarray(x, np.int64)
        out = np.full((x.shape[0], x.shape[1] + 1), -1, np.int64)
        for b in range(x.shape[0]):
            out[b, :int(n_accept[b])] = x[b, :int(n_accept[b])]
        return out
    monkeypatch.setattr(R, "emitted_tokens", bad)
    assert _fails(T_rounds.test_anchor_is_the_last_emitted_token)
    assert _fails(T_rounds.test_agreeing_target_accepts_every_scheduled_token)


def test_heads_inverted_gate_is_caught(monkeypatch):
    from oracle import heads as Hd
    import tests.test_oracle_heads as T_heads
    orig = Hd.sigmoid
    monkeypatch.setattr(Hd, "sigmoid", lambda x: 1.0 - orig(x))
    assert _fails(T_heads.test_saturated_gates_reduce_to_closed_forms)


def test_heads_state_not_carried_is_caught(monkeypatch):
    from oracle import heads as Hd
    import tests.test_oracle_heads as T_heads
    orig = Hd.Head.step
    monkeypatch.setattr(Hd.Head, "step", lambda self, W1p, hk, st: orig(self, W1p, hk, np.zeros_like(st)))
    assert _fails(T_heads.test_rnn_half_gate_is_the_unrolled_sum)


def test_heads_gate_on_the_next_hidden_state_is_caught(monkeypatch):
    from oracle import heads as Hd
    import tests.test_oracle_heads as T_heads
    orig = Hd.Head.step
    monkeypatch.setattr(Hd.Head, "step", lambda self, W1p, hk, st: orig(self, W1p, np.roll(hk, 1, axis=0), st))
    assert _fails(T_heads.test_gate_reads_h_of_its_own_position)


def test_residual_rebuilt_from_the_wrong_previous_token_is_caught(monkeypatch):
    # the rejected row's draft logits rebuilt with x_k in place of x_{k-1} (for k = 1: x_1, not the anchor)
    import oracle.verify as V
    orig = V.draft_logits

    def bad(U, W1, W2, x0, tokens, b, k, E=None):
        t = np.asarray(tokens)
        return orig(U, W1, W2, t[:, 0], t, b, k, E=E)
    monkeypatch.setattr(V, "draft_logits", bad)
    assert _fails(T_verify.test_token_after_a_rejection_follows_the_residual)


def test_temperature_on_the_base_logits_only_is_caught(monkeypatch):
    # l = U / T + B instead of (U + B) / T: the bias scaled by T before the division
    orig = draft.markov_bias
    T = 0.8                                                   # the strong-bias test's temperature
    monkeypatch.setattr(draft, "markov_bias", lambda W1, W2, prev: T * orig(W1, W2, prev))
    assert _fails(T_draft.test_draft_sample_distribution_with_strong_bias)


def test_expected_tokens_without_the_bonus_token_is_caught(monkeypatch):
    # E = sum of the scheduled survivals only, dropping each request's certain token
    # (reading 3: E = sum_b (1 + sum_{j <= l_b} a_{b,j}))
    from fractions import Fraction

    def bad(a, sps):
        a = np.asarray(a, np.float32)
        B, G = a.shape
        pairs = sorted(((b, j) for b in range(B) for j in range(1, G + 1)),
                       key=lambda p: (-float(a[p[0], p[1] - 1]), p[0], p[1]))
        ell, E, N = np.zeros(B, np.int64), Fraction(0), B
        best = float(E) / N * sps[N]
        for b, j in pairs:
            E_new = E + Fraction(float(a[b, j - 1]))
            th = float(E_new) / (N + 1) * sps[N + 1]
            if th > best:
                ell[b] += 1
                E, N, best = E_new, N + 1, th
            else:
                break
        return ell, N, best
    monkeypatch.setattr(schedule, "schedule_prefix", bad)
    assert _fails(T_sched.test_greedy_stop_is_global_optimum_for_rational_sps)


def test_philox_swapped_multipliers_are_caught(monkeypatch):
    import tests.test_oracle_philox as T_philox
    monkeypatch.setattr(philox, "_M0", philox._M1)
    monkeypatch.setattr(philox, "_M1", philox._M0)
    assert _fails(lambda: [T_philox.test_known_answer_vectors(r) for r in T_philox._kat_rows()])


def test_philox_missing_key_bump_is_caught(monkeypatch):
    import tests.test_oracle_philox as T_philox
    monkeypatch.setattr(philox, "_W1", np.uint64(0))
    assert _fails(lambda: [T_philox.test_known_answer_vectors(r) for r in T_philox._kat_rows()])


def test_loss_position_weight_off_by_one_is_caught(monkeypatch):
    # exp(-k / gamma) instead of exp(-(k - 1) / gamma): the first position no longer weighs 1
    from oracle import loss as L
    import tests.test_oracle_loss as T_loss
    monkeypatch.setattr(L, "position_weights",
                        lambda k, decay=L.DECAY_GAMMA: np.exp(-np.asarray(k, np.float64) / decay))
    assert _fails(T_loss.test_position_weights)
