"""fp64 CPU oracle of the Goldfish-loss masked cross-entropy.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may load it.  It
shares no code with the CUDA path (which implements the same hash from the
same published definition, separately).

What it follows
---------------
* The pith.science review of arXiv 2502.08145, "What carries the argument":
  against memorisation the paper trains with Goldfish Loss, which masks
  tokens at random so that the cross-entropy loss is not computed on them.
* The same review, "Assumptions & free parameters": the mask parameters are
  k = 2 and h = 13.  The pages cite the method's own paper (Hans et al., "Be
  like a Goldfish, Don't Memorize!", arXiv 2406.10209) for it: one token in
  k is left out of the loss, and the choice is a hash of the h tokens that
  precede it, so a passage seen twice is masked the same way both times.

Readings where the pages are silent (each also listed in the design notes)
--------------------------------------------------------------------------
1. Sequences are rows of ``input_ids`` [B x S]; ``labels`` [B x S] holds the
   token each position predicts (the next token).  The window of label
   (b, t) is the h input tokens ending at position t, input_ids[b, t-h+1 ..
   t] -- the h tokens that precede the label in the document.  Windows never
   cross rows.
2. The hash H is 64-bit FNV-1a (Fowler, Noll and Vo; offset basis
   0xcbf29ce484222325, prime 0x100000001b3) over the window's token ids,
   each written as 4 little-endian bytes, oldest first.  Label (b, t) is
   dropped when H mod k == 0, so on average one in k labels is dropped.
3. A label with fewer than h tokens before it (t < h - 1) has no full
   window and is kept.
4. k = 0 turns the mask off (plain cross-entropy); k = 1 drops every label
   that has a full window.  A label outside [0, V) is padding: never
   counted.
5. Cross-entropy of position t: CE_t = logsumexp(z_t) - z_t[y_t] over the
   row of logits z_t (natural log).  The loss is the mean over kept labels,
   sum_t G_t CE_t / n, n = sum_t G_t (G_t = 1 for a kept label); with n = 0
   the loss is 0.  Its gradient with respect to the logits is
   G_t (softmax(z_t) - e_{y_t}) / n (zero rows for dropped labels).

Parity: the mask (integers) is exact; the fp64 values here bound the
kernel's fp32 ones as stated in the GPU tests.  Pins: tests/test_goldfish.py
(FNV-1a's published test vectors, hand-worked cross-entropy, the mask-off
case against torch's cross-entropy and its autograd gradient, k = 1, the
invariants of a hashed mask).
"""
from __future__ import annotations

import numpy as np

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a of a byte string: for each byte, xor it into the state,
    then multiply by the prime modulo 2^64."""
    h = FNV_OFFSET
    for byte in data:
        h = ((h ^ byte) * FNV_PRIME) & MASK64
    return h


def window_bytes(window) -> bytes:
    """Token ids of one window as 4 little-endian bytes each, oldest first."""
    return b"".join(int(t & 0xFFFFFFFF).to_bytes(4, "little") for t in window)


def goldfish_keep(input_ids: np.ndarray, labels: np.ndarray, k: int, h: int,
                  vocab: int | None = None) -> np.ndarray:
    """G[b, t] in {0, 1}: 1 where label (b, t) counts in the loss (labels
    below 0, or at or above `vocab` when given, are padding)."""
    ids = np.asarray(input_ids, dtype=np.int64)
    lab = np.asarray(labels, dtype=np.int64)
    assert ids.shape == lab.shape and ids.ndim == 2 and k >= 0 and h >= 1
    B, S = ids.shape
    keep = np.zeros((B, S), dtype=np.uint8)
    for b in range(B):
        for t in range(S):
            if lab[b, t] < 0 or (vocab is not None and lab[b, t] >= vocab):
                continue                      # padding
            if k == 0 or t < h - 1:
                keep[b, t] = 1                # mask off, or no full window
                continue
            H = fnv1a64(window_bytes(ids[b, t - h + 1: t + 1]))
            keep[b, t] = 0 if H % k == 0 else 1
    return keep


def _logits_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def cross_entropy_rows(logit_bits: np.ndarray, labels_flat: np.ndarray):
    """CE_t = logsumexp(z_t) - z_t[y_t] and the softmax of each row, fp64;
    rows whose label is below 0 give CE 0."""
    z = _logits_f64(logit_bits)
    y = np.asarray(labels_flat, dtype=np.int64)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    s = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(s))[:, 0]
    p = e / s
    ce = np.zeros(z.shape[0])
    ok = y >= 0
    ce[ok] = lse[ok] - z[np.nonzero(ok)[0], y[ok]]
    return ce, p, lse


def goldfish_ce(logit_bits, input_ids, labels, k: int, h: int, rows=None):
    """Goldfish-masked cross-entropy.

    logit_bits: bf16 bits [B*S x V] (uint16), one row per position in
    row-major (b, t) order.  Returns dict with
      keep [B*S] u8, n (kept labels), loss (mean over kept, 0 if none),
      token_loss [B*S] (CE_t for kept labels, 0 otherwise),
      and, for the positions in `rows` (default all), dlogits [len(rows) x V]
      = G_t (softmax(z_t) - e_{y_t}) / n.
    With `rows` given, only those rows of `logit_bits` are read (pass the
    rows themselves as logit_bits); loss and token_loss then cover only
    them, while keep and n still cover every position."""
    ids = np.asarray(input_ids)
    lab = np.asarray(labels)
    keep = goldfish_keep(ids, lab, k, h, vocab=np.shape(logit_bits)[1]).reshape(-1)
    n = int(keep.sum())
    y = lab.reshape(-1).astype(np.int64)
    idx = np.arange(y.size) if rows is None else np.asarray(rows, dtype=np.int64)
    ce, p, lse = cross_entropy_rows(logit_bits, np.where(keep[idx] == 1, y[idx], -1))
    token_loss = np.where(keep[idx] == 1, ce, 0.0)
    grad = np.zeros_like(p)
    if n > 0:
        kept_rows = np.nonzero(keep[idx])[0]
        grad[kept_rows] = p[kept_rows]
        grad[kept_rows, y[idx][kept_rows]] -= 1.0
        grad /= n
    loss = float(token_loss.sum() / n) if n > 0 else 0.0
    return {"keep": keep, "n": n, "loss": loss, "token_loss": token_loss,
            "dlogits": grad, "lse": lse, "softmax": p}


def goldfish_loss_streamed(get_rows, input_ids, labels, k: int, h: int, vocab: int,
                           chunk: int = 256):
    """The Goldfish loss over logits too large to hold in fp64 at once:
    get_rows(r0, r1) returns bf16 bits of logit rows [r0, r1).  Returns
    (loss, n, token_loss [T], keep [T]); rows of dropped labels are not
    requested."""
    ids = np.asarray(input_ids)
    lab = np.asarray(labels)
    keep = goldfish_keep(ids, lab, k, h, vocab=vocab).reshape(-1)
    y = lab.reshape(-1).astype(np.int64)
    T = y.size
    token_loss = np.zeros(T)
    for r0 in range(0, T, chunk):
        r1 = min(T, r0 + chunk)
        if not keep[r0:r1].any():
            continue
        ce, _, _ = cross_entropy_rows(get_rows(r0, r1), np.where(keep[r0:r1] == 1, y[r0:r1], -1))
        token_loss[r0:r1] = np.where(keep[r0:r1] == 1, ce, 0.0)
    n = int(keep.sum())
    loss = float(token_loss.sum() / n) if n > 0 else 0.0
    return loss, n, token_loss, keep
