"""Algorithmic FLOPs and compulsory HBM bytes of the chunked gated delta rule.

FLOPs count what the chunk algorithm itself must compute (2 per multiply-add), per chunk of
c tokens, d = K = V:
  forward,  per (chunk, q/k head):  Q K^T and K K^T               2 * 2 c^2 d
            per (chunk, v head):    T Y_W, T Y_U, P V'            3 * 2 c^2 d
                                    W h, diag(e) Q h, Khat^T V'   3 * 2 c d^2
                                    the triangular inverse        c^3 / 3
  backward, per (chunk, q/k head):  dS K, dS^T Q, (dB + dB^T) K   3 * 2 c^2 d
            per (chunk, v head):    6 * 2 c^2 d + 6 * 2 c d^2 + 2 * 2 c^3
Context-parallel overheads (segment transitions, fix-up, rerun) and the backward's
recompute are implementation choices and are not counted.

Bytes are compulsory traffic: every input read once and every output written once.
"""
from __future__ import annotations


def _chunk_lengths(lengths, C):
    for L in lengths:
        full, rem = divmod(L, C)
        for _ in range(full):
            yield C
        if rem:
            yield rem


def fwd_flops(lengths, Hqk, Hv, d=128, C=64):
    f = 0.0
    for c in _chunk_lengths(lengths, C):
        f += Hqk * 2 * 2 * c * c * d
        f += Hv * (3 * 2 * c * c * d + 3 * 2 * c * d * d + c ** 3 / 3)
    return f


def bwd_flops(lengths, Hqk, Hv, d=128, C=64):
    f = 0.0
    for c in _chunk_lengths(lengths, C):
        f += Hqk * 3 * 2 * c * c * d
        f += Hv * (6 * 2 * c * c * d + 6 * 2 * c * d * d + 2 * 2 * c ** 3)
    return f


def fwd_bytes(T_total, N, Hqk, Hv, d=128, elem=2, h0=False, ht=True):
    b = 2 * T_total * Hqk * d * elem          # q, k
    b += T_total * Hv * d * elem              # v
    b += 2 * T_total * Hv * 4                 # g, beta
    b += T_total * Hv * d * elem              # o
    state = N * Hv * d * d * 4
    b += state * (int(h0) + int(ht))
    return float(b)


def bwd_bytes(T_total, N, Hqk, Hv, d=128, elem=2, h0=True, dht=True):
    b = 2 * T_total * Hqk * d * elem          # q, k
    b += 2 * T_total * Hv * d * elem          # v, dO
    b += 2 * T_total * Hv * 4                 # g, beta
    b += 2 * T_total * Hqk * d * elem         # dq, dk
    b += T_total * Hv * d * elem              # dv
    b += 2 * T_total * Hv * 4                 # dg, dbeta
    state = N * Hv * d * d * 4
    b += state * (int(h0) + int(dht) + int(h0))  # h0, dht, dh0
    return float(b)
