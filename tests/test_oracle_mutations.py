"""Plant plausible mistakes in the oracle (on the CPU, in a patched copy of its functions)
and check that at least one pin catches each.  This is what makes the pins worth trusting:
a dropped term, a wrong sign, a wrong axis or a transposed operand must not pass."""
import math

import numpy as np
import pytest

import oracle.attnres_oracle as O
import oracle_pins


def _rms_sum(x, eps):                       # forgets the 1/d of the mean
    x = np.asarray(x, np.float64)
    return np.sqrt(np.sum(x * x, axis=-1) + eps)


def _rms_no_eps(x, eps):                    # drops eps
    x = np.asarray(x, np.float64)
    return np.sqrt(np.mean(x * x, axis=-1))


def _rms_centered(x, eps):                  # LayerNorm-style variance instead of m_2
    x = np.asarray(x, np.float64)
    return np.sqrt(np.var(x, axis=-1) + eps)


def _softmax_neg(z):                        # wrong sign in the exponent
    z = np.asarray(z, np.float64)
    e = np.exp(-(z - np.min(z, axis=0, keepdims=True)))
    return e / e.sum(axis=0, keepdims=True)


def _softmax_wrong_axis(z):                 # normalises over tokens instead of sources
    z = np.asarray(z, np.float64)
    e = np.exp(z - np.max(z, axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _logits_scaled(sources, w, gamma_key, eps):   # adds a 1/sqrt(d) scale the pages do not have
    keys = O.rmsnorm(sources, gamma_key, eps)
    return np.sum(keys * np.asarray(w, np.float64), axis=-1) / math.sqrt(np.shape(sources)[-1])


def _logits_raw_keys(sources, w, gamma_key, eps):  # forgets the key RMSNorm
    src = np.asarray(sources, np.float64)
    g = 1.0 if gamma_key is None else np.asarray(gamma_key, np.float64)
    return np.sum(src * g * np.asarray(w, np.float64), axis=-1)


def _logits_gamma_on_query_index_reversed(sources, w, gamma_key, eps):  # transposed gain
    keys = O.rmsnorm(sources, None if gamma_key is None else np.asarray(gamma_key)[::-1], eps)
    return np.sum(keys * np.asarray(w, np.float64), axis=-1)


def _aggregate_normed_values(sources, w, gamma_key, eps):  # uses keys as values
    src = np.asarray(sources, np.float64)
    z = O.depth_logits(src, w, gamma_key, eps)
    alpha = O.depth_softmax(z)
    return np.sum(alpha[..., None] * O.rmsnorm(src, None, eps), axis=0), alpha, z


def _partition_lse_no_max(sources, w, gamma_key, eps):  # returns ln l instead of m + ln l
    o, m, lse, a = _ORIG_PARTITION(sources, w, gamma_key, eps)
    return o, m, lse - m, a


def _partition_unnormalised(sources, w, gamma_key, eps):  # forgets to divide o by l
    o, m, lse, a = _ORIG_PARTITION(sources, w, gamma_key, eps)
    return o * np.exp(lse - m)[..., None], m, lse, a


def _block_sources_zero_partial(completed, partial):  # a zero source at the first sublayer
    srcs = [np.asarray(b, np.float64) for b in completed]
    srcs.append(np.zeros_like(srcs[0]) if partial is None else np.asarray(partial, np.float64))
    return np.stack(srcs)


def _block_of_off_by_one(l, S):             # blocks start one sublayer late
    n = l // S + 1
    return n, l - (n - 1) * S + 1


def _merge_ignores_lse(o_A, lse_A, p, w, gamma_key, eps_key, gamma_in, eps_in):  # drops e^{lse}
    h, y, a = _ORIG_MERGE(o_A, np.zeros_like(np.asarray(lse_A, np.float64)), p, w, gamma_key,
                          eps_key, gamma_in, eps_in)
    return h, y, a


def _sigmoid_normalised(z):                 # sigmoid weights divided by their sum
    a = 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))
    return a / a.sum(axis=0, keepdims=True)


def _sigmoid_sign(z):                       # sigmoid of -z
    return 1.0 / (1.0 + np.exp(np.asarray(z, np.float64)))


def _raw_logits_still_normalised(sources, w):  # "no key norm" that still divides by r
    src = np.asarray(sources, np.float64)
    return np.sum(src / O.rms(src, 0.0)[..., None] * np.asarray(w, np.float64), axis=-1)


def _merge_variant_softmax_for_sigmoid(o_A, lse_A, p, w, gamma_key, eps_key, gamma_in, eps_in,
                                       weights="softmax", key_norm=True):
    # merges sigmoid partitions as if they were softmax partitions (lse taken as 0)
    lse = np.zeros(np.shape(o_A)[:-1]) if lse_A is None else lse_A
    return _ORIG_MERGE_V(o_A, lse, p, w, gamma_key, eps_key, gamma_in, eps_in, "softmax",
                         key_norm)


def _merge_sources_drops_history(o_A, lse_A, sources_B, w, gamma_key, eps_key, gamma_in,
                                 eps_in):               # forgets partition A's exp-sum weight
    h, y, aB, wA = _ORIG_MERGE_S(o_A, np.full_like(np.asarray(lse_A, np.float64), -50.0),
                                 sources_B, w, gamma_key, eps_key, gamma_in, eps_in)
    return h, y, aB, wA


def _rmsnorm_backward_no_radial(x, gamma, eps, g):   # drops the radial correction term
    x, g = np.asarray(x, np.float64), np.asarray(g, np.float64)
    r = O.rms(x, eps)[..., None]
    gp = g if gamma is None else g * np.asarray(gamma, np.float64)
    return gp / r, g * x / r


def _aggregate_backward_no_minus_h(sources, w, gamma_key, eps_key, gamma_in, eps_in, g_y):
    # logit gradient alpha_i g^T v_i, without the - h of page 2 §7
    G = _ORIG_BACKWARD(sources, w, gamma_key, eps_key, gamma_in, eps_in, g_y)
    v = np.asarray(sources, np.float64)
    _, alpha, _ = O.aggregate(v, w, gamma_key, eps_key)
    dz_bad = alpha * np.sum(G.g_h[None] * v, axis=-1)
    keys = O.rmsnorm(v, gamma_key, eps_key)
    G.dw = np.sum(dz_bad[..., None] * keys, axis=(0, 1))
    G.dz = dz_bad
    return G


def _head_slices_interleaved(d, H):        # head k takes every H-th feature instead of a block
    assert d % H == 0
    return [slice(k, d, H) for k in range(H)]


def _multihead_row_norm(sources, w, gamma_key, eps, H, weights="softmax", key_norm=True):
    # the key RMS over the whole row instead of the head's slice
    src = np.asarray(sources, np.float64)
    d = src.shape[-1]
    r = O.rms(src, eps)[..., None]
    h = np.zeros(src.shape[1:])
    al, zz = [], []
    for sl in O.head_slices(d, H):
        g = 1.0 if gamma_key is None else np.asarray(gamma_key, np.float64)[sl]
        z = np.sum(np.asarray(w, np.float64)[sl] * g * src[..., sl] / r, axis=-1)
        a = O.depth_softmax(z)
        h[..., sl] = np.sum(a[..., None] * src[..., sl], axis=0)
        al.append(a)
        zz.append(z)
    return h, np.stack(al), np.stack(zz)


def _block_backward_partial_off_by_one(completed, v, W, G_key, G_in, eps_key, eps_in, g_y):
    # hands the partial gradient of sublayer i to v_1 .. v_i instead of v_1 .. v_{i-1}
    G = _ORIG_BLOCK_BACKWARD(completed, v, W, G_key, G_in, eps_key, eps_in, g_y)
    S = G.dv.shape[0]
    G.dv = np.stack([G.dpartial[k:].sum(axis=0) for k in range(S)])
    return G


_ORIG_BLOCK_BACKWARD = O.block_backward
_ORIG_PARTITION = O.partition_stats
_ORIG_BACKWARD = O.aggregate_backward
_ORIG_MERGE_S = O.merge_sources_reference
_ORIG_MERGE_V = O.merge_reference_variant
_ORIG_MERGE = O.merge_reference

MUTATIONS = {
    "rms_sum_not_mean": ("rms", _rms_sum),
    "rms_drops_eps": ("rms", _rms_no_eps),
    "rms_centered": ("rms", _rms_centered),
    "softmax_sign": ("depth_softmax", _softmax_neg),
    "softmax_axis": ("depth_softmax", _softmax_wrong_axis),
    "logit_scale": ("depth_logits", _logits_scaled),
    "no_key_norm": ("depth_logits", _logits_raw_keys),
    "gain_transposed": ("depth_logits", _logits_gamma_on_query_index_reversed),
    "normed_values": ("aggregate", _aggregate_normed_values),
    "lse_without_max": ("partition_stats", _partition_lse_no_max),
    "o_unnormalised": ("partition_stats", _partition_unnormalised),
    "zero_partial_source": ("block_sources", _block_sources_zero_partial),
    "block_index_off_by_one": ("block_of", _block_of_off_by_one),
    "merge_ignores_lse": ("merge_reference", _merge_ignores_lse),
    "sigmoid_normalised": ("depth_sigmoid", _sigmoid_normalised),
    "sigmoid_sign": ("depth_sigmoid", _sigmoid_sign),
    "raw_logits_normalised": ("depth_logits_raw", _raw_logits_still_normalised),
    "sigmoid_merged_as_softmax": ("merge_reference_variant", _merge_variant_softmax_for_sigmoid),
    "merge_sources_drops_history": ("merge_sources_reference", _merge_sources_drops_history),
    "rmsnorm_backward_no_radial": ("rmsnorm_backward", _rmsnorm_backward_no_radial),
    "logit_gradient_without_h": ("aggregate_backward", _aggregate_backward_no_minus_h),
    "block_backward_partial_off_by_one": ("block_backward", _block_backward_partial_off_by_one),
    "heads_interleaved": ("head_slices", _head_slices_interleaved),
    "head_key_norm_over_row": ("multihead_aggregate", _multihead_row_norm),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(O, attr, bad)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake {name}"
