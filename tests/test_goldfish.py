"""Pins of the Goldfish-loss oracle (oracle/goldfish.py), on the CPU, against
things other than itself:

* FNV-1a's published 64-bit test vectors, and a window's byte string
  written out by hand;
* hand-worked cross-entropy values;
* with the mask off (k = 0) the loss and its gradient equal torch's
  cross-entropy and torch's autograd gradient (a library special case);
  with the mask on they equal torch's cross-entropy with the dropped labels
  set to its ignore index (the composition of mask and mean);
* k = 1 drops every label with a full window; labels without one are kept;
* the hashed mask's invariants: the decision depends only on the window,
  identical windows decide alike, and about one label in k is dropped;
* a planted mistake (normalising by every label instead of the kept ones)
  is caught.
"""
import numpy as np
import pytest

import fc_inputs
from oracle import goldfish as gf


def test_fnv1a64_published_vectors():
    # Fowler-Noll-Vo test vectors for 64-bit FNV-1a
    assert gf.fnv1a64(b"") == 0xCBF29CE484222325
    assert gf.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert gf.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_window_bytes_by_hand():
    assert gf.window_bytes([1, 256, 0x01020304]) == bytes(
        [1, 0, 0, 0, 0, 1, 0, 0, 4, 3, 2, 1])


def test_mask_decision_from_hand_written_bytes():
    """Sequence 5, 7, 9 with h = 2: label 0 has no full window (kept); label
    1's window is (5, 7), label 2's is (7, 9), hashed from their bytes
    written out here."""
    ids = np.array([[5, 7, 9]])
    labels = np.array([[7, 9, 11]])
    h57 = gf.fnv1a64(bytes([5, 0, 0, 0, 7, 0, 0, 0]))
    h79 = gf.fnv1a64(bytes([7, 0, 0, 0, 9, 0, 0, 0]))
    for k in (2, 3, 5, 7):
        keep = gf.goldfish_keep(ids, labels, k, 2)
        assert keep.tolist() == [[1, int(h57 % k != 0), int(h79 % k != 0)]]


def _bits(a):
    return fc_inputs.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_cross_entropy_hand_values():
    # uniform row of 3: CE = ln 3 for every label
    ce, _, _ = gf.cross_entropy_rows(_bits([[0.5, 0.5, 0.5]] * 3), np.array([0, 1, 2]))
    assert np.allclose(ce, 1.0986122886681098, rtol=0, atol=1e-15)
    # logits 0, 1, 2, label 2: ln(1 + e^-1 + e^-2) = ln(1.5032147244...) = 0.4076059644...
    # label 0: 2 + 0.4076059644 = 2.4076059644
    ce, p, lse = gf.cross_entropy_rows(_bits([[0.0, 1.0, 2.0]] * 2), np.array([2, 0]))
    assert abs(ce[0] - 0.40760596444438) < 1e-12
    assert abs(ce[1] - 2.40760596444438) < 1e-12
    # softmax of 0, 1, 2: 1, e, e^2 over 11.1073379... = 0.0900306, 0.2447285, 0.6652410
    assert np.allclose(p[0], [0.09003057317038, 0.24472847105479, 0.66524095577483], atol=1e-12)
    # a dominant logit: CE of the dominant label is about 2 e^-30
    ce, _, _ = gf.cross_entropy_rows(_bits([[0.0, 0.0, 30.0]] * 2), np.array([2, 0]))
    assert 0 < ce[0] < 2e-13 and abs(ce[1] - 30.0) < 1e-12


def _problem(B, S, V, seed, pad_every=0):
    rng = np.random.default_rng(seed)
    seqs = rng.integers(0, V, size=(B, S + 1))
    ids, labels = seqs[:, :-1].copy(), seqs[:, 1:].copy()
    if pad_every:
        labels[:, ::pad_every] = -100
    logits = fc_inputs.normal_bf16((B * S, V), seed, 7, sigma=2.0)
    return ids, labels, logits


def _torch_reference(logits_bits, labels_flat):
    torch = pytest.importorskip("torch")
    z = torch.tensor(fc_inputs.bf16_bits_to_f32(logits_bits), dtype=torch.float64,
                     requires_grad=True)
    y = torch.tensor(labels_flat, dtype=torch.int64)
    if (y >= 0).sum() == 0:
        return 0.0, np.zeros(z.shape)
    loss = torch.nn.functional.cross_entropy(z, y, ignore_index=-100, reduction="mean")
    loss.backward()
    return float(loss.detach()), z.grad.numpy()


@pytest.mark.parametrize("B,S,V,pad", [(2, 7, 11, 0), (3, 20, 50, 3), (1, 40, 300, 0)])
def test_mask_off_is_plain_cross_entropy(B, S, V, pad):
    ids, labels, logits = _problem(B, S, V, 31 + V, pad_every=pad)
    out = gf.goldfish_ce(logits, ids, labels, k=0, h=13)
    assert out["n"] == int((labels >= 0).sum())
    loss, grad = _torch_reference(logits, labels.reshape(-1))
    assert abs(out["loss"] - loss) <= 1e-12 * max(1.0, abs(loss))
    assert np.allclose(out["dlogits"], grad, rtol=0, atol=1e-14)


@pytest.mark.parametrize("k,h", [(2, 13), (2, 1), (3, 4), (4, 13)])
def test_masked_loss_is_cross_entropy_over_kept_labels(k, h):
    """Goldfish loss = torch's mean cross-entropy with the dropped labels
    set to the ignore index; gradient = torch's autograd gradient."""
    ids, labels, logits = _problem(4, 32, 97, 40 + k * h, pad_every=5)
    out = gf.goldfish_ce(logits, ids, labels, k=k, h=h)
    masked = np.where(out["keep"] == 1, labels.reshape(-1), -100)
    loss, grad = _torch_reference(logits, masked)
    assert 0 < out["n"] < (labels >= 0).sum()
    assert abs(out["loss"] - loss) <= 1e-12 * max(1.0, abs(loss))
    assert np.allclose(out["dlogits"], grad, rtol=0, atol=1e-14)
    # dropped and padded positions contribute nothing
    assert np.all(out["token_loss"][out["keep"] == 0] == 0)
    assert np.all(out["dlogits"][out["keep"] == 0] == 0)


def test_k1_drops_every_label_with_a_full_window():
    ids, labels, logits = _problem(2, 30, 40, 51)
    h = 13
    out = gf.goldfish_ce(logits, ids, labels, k=1, h=h)
    keep = out["keep"].reshape(2, 30)
    assert np.all(keep[:, : h - 1] == 1) and np.all(keep[:, h - 1:] == 0)
    assert out["n"] == 2 * (h - 1)
    loss, _ = _torch_reference(logits, np.where(out["keep"] == 1, labels.reshape(-1), -100))
    assert abs(out["loss"] - loss) < 1e-12
    # nothing kept at all: loss 0, gradient 0
    out = gf.goldfish_ce(logits, ids, np.full_like(labels, -100), k=2, h=h)
    assert out["n"] == 0 and out["loss"] == 0.0 and not np.any(out["dlogits"])


def test_hashed_mask_invariants():
    rng = np.random.default_rng(61)
    V, h = 50000, 13
    ids = rng.integers(0, V, size=(4, 2500))
    labels = rng.integers(0, V, size=(4, 2500))
    # about one label in k is dropped (binomial, 10^4 labels: 0.5 +- 0.015)
    for k, lo, hi in ((2, 0.47, 0.53), (4, 0.22, 0.28)):
        keep = gf.goldfish_keep(ids, labels, k, h)
        frac = 1 - keep[:, h - 1:].mean()
        assert lo < frac < hi, (k, frac)
    # the decision depends only on the window: change tokens outside it
    keep = gf.goldfish_keep(ids, labels, 2, h)
    ids2 = ids.copy()
    ids2[:, :100] = rng.integers(0, V, size=(4, 100))
    keep2 = gf.goldfish_keep(ids2, labels, 2, h)
    assert np.array_equal(keep[:, 100 + h - 1:], keep2[:, 100 + h - 1:])
    # identical windows decide alike (a passage seen twice is masked alike)
    rep = np.concatenate([ids[:1, :300], ids[:1, :300]], axis=1)
    krep = gf.goldfish_keep(rep, np.zeros_like(rep), 2, h)
    assert np.array_equal(krep[0, h - 1:300], krep[0, 300 + h - 1:])
    # and windows are ordered: reversing a window changes its hash
    w = [11, 22, 33]
    assert gf.fnv1a64(gf.window_bytes(w)) != gf.fnv1a64(gf.window_bytes(w[::-1]))


def test_planted_mistake_is_caught(monkeypatch):
    """A loss averaged over every label instead of the kept ones fails the
    torch pin."""
    ids, labels, logits = _problem(4, 32, 97, 77)
    real = gf.goldfish_ce

    def wrong(*a, **kw):
        out = real(*a, **kw)
        out["loss"] = float(out["token_loss"].sum() / out["keep"].size)
        return out

    monkeypatch.setattr(gf, "goldfish_ce", wrong)
    out = gf.goldfish_ce(logits, ids, labels, k=2, h=13)
    loss, _ = _torch_reference(logits, np.where(out["keep"] == 1, labels.reshape(-1), -100))
    assert abs(out["loss"] - loss) > 1e-3


def test_rows_subset_matches_whole():
    ids, labels, logits = _problem(2, 24, 64, 81)
    whole = gf.goldfish_ce(logits, ids, labels, 2, 13)
    rows = np.array([0, 5, 17, 30, 47])
    part = gf.goldfish_ce(logits[rows], ids, labels, 2, 13, rows=rows)
    assert part["n"] == whole["n"]
    assert np.array_equal(part["token_loss"], whole["token_loss"][rows])
    assert np.array_equal(part["dlogits"], whole["dlogits"][rows])


def test_streamed_loss_matches_whole():
    ids, labels, logits = _problem(3, 50, 80, 91)
    whole = gf.goldfish_ce(logits, ids, labels, 2, 13)
    loss, n, tl, keep = gf.goldfish_loss_streamed(lambda a, b: logits[a:b], ids, labels, 2, 13,
                                                  vocab=80, chunk=17)
    assert n == whole["n"] and np.array_equal(keep, whole["keep"])
    assert np.array_equal(tl, whole["token_loss"]) and loss == whole["loss"]


def test_labels_outside_the_vocabulary_are_padding():
    ids, labels, logits = _problem(2, 20, 30, 95)
    labels[0, 3] = 30
    labels[1, 7] = 1000
    out = gf.goldfish_ce(logits, ids, labels, 0, 13)
    assert out["keep"].reshape(2, 20)[0, 3] == 0 and out["keep"].reshape(2, 20)[1, 7] == 0
    assert out["n"] == 38
