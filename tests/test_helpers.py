"""The parity helpers themselves (CPU): a block check finds one wrong chunk, one
wrong sequence or one wrong boundary row that the whole-tensor relative L2 misses."""
import numpy as np

from tests import helpers as H


def _tensors(rng, lens, H_=2, D=16):
    T = sum(lens)
    ref = rng.standard_normal((T, H_, D))
    gpu = ref * (1 + 1e-3 * rng.standard_normal(ref.shape))  # a correct result: small relative noise
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return gpu, ref, cu


def test_block_errors_of_a_correct_result_are_small():
    rng = np.random.default_rng(0)
    gpu, ref, cu = _tensors(rng, [1, 63, 64, 65, 600])
    ws, wc, wr = H.block_errors(gpu, ref, cu)
    assert max(ws, wc, wr) < 5e-3
    assert H.rel_l2(gpu, ref) < 2e-3


def test_one_unwritten_chunk_fails_the_chunk_check_only():
    rng = np.random.default_rng(1)
    gpu, ref, cu = _tensors(rng, [100000, 70000], D=4)
    gpu[64 * 7:64 * 8, 1] = 0.0  # one chunk of one head left unwritten
    assert H.rel_l2(gpu, ref) < H.TOL_BF16  # diluted below the tolerance in the whole tensor
    ws, wc, wr = H.block_errors(gpu, ref, cu)
    assert wc > 0.9 and wc > H.BLOCK_TOL_FACTOR * H.TOL_BF16 and wc > ws


def test_a_wrong_boundary_row_fails_the_row_check():
    rng = np.random.default_rng(2)
    gpu, ref, cu = _tensors(rng, [300, 77, 5000])
    gpu[376] = 0.0  # the last valid row of the second sequence left unwritten
    assert H.rel_l2(gpu, ref) < 2e-2
    ws, wc, wr = H.block_errors(gpu, ref, cu)
    assert wr > 0.9


def test_vanishing_blocks_are_floored():
    rng = np.random.default_rng(3)
    gpu, ref, cu = _tensors(rng, [64, 64])
    ref[64:] *= 1e-2  # a block whose true values nearly cancel ...
    gpu[64:] = ref[64:] + 1e-5 * rng.standard_normal(ref[64:].shape)  # ... computed to 1e-3 of its own size
    ws, wc, wr = H.block_errors(gpu, ref, cu)
    assert ws < 2e-3  # judged against the average magnitude, not its own (which would give ~1e-3 too)
