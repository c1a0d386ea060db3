"""rq_validate_indices_noalloc: the index check for callers that cannot
allocate device memory (a program with no device allocator of its own, or an
engine that has given all free memory to its KV cache). It keeps its scratch in
a fixed device array of the library instead of a caller workspace.

This file is collected last, so a run that stops at its first failure has
already run every other test. It passes alone in a fresh process and after the
other tests: the array keeps the previous call's bits, and each call must
clear what it uses, which the second call of each pair below checks.
"""
import ctypes

import pytest
import torch

import rope_block_fp8_inverse_b300 as rq
import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(pos, slots, cache_rows, num_slots):
    out = ctypes.c_uint32(0xDEAD)
    st = rq.lib().rq_validate_indices_noalloc(
        pos.data_ptr(), 0 if slots is None else slots.data_ptr(), pos.shape[0], cache_rows,
        num_slots, ctypes.addressof(out), torch.cuda.current_stream().cuda_stream)
    assert st == 0, rq.status_string(st)
    return out.value


def test_noalloc_check_matches_the_workspace_entry_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    ins = W.insert_inputs(W.INSERT16K)
    pos, slots = ins["positions"].to(dev), ins["slot_mapping"].to(dev)
    n_slots = W.INSERT16K.num_blocks * W.INSERT16K.block_size
    dup = slots.clone()
    dup[100] = dup[7]                                   # one slot written twice
    bad = torch.tensor([0, 5, 70000, 3], device=dev)    # one position past the cache
    cases = [(pos, dup, 65536, n_slots), (pos, slots, 65536, n_slots),   # dirty, then clean
             (bad, None, 65536, 0), (pos, slots, 65536, n_slots)]
    for p_, s_, rows, ns in cases:
        want = rq.validate_indices(p_, rows, s_, ns)
        assert _noalloc(p_, s_, rows, ns) == want
    assert rq.validate_indices(pos, 65536, dup, n_slots) == 8


def test_noalloc_check_rejects_more_slots_than_its_array_holds():
    dev = torch.device("cuda:0")
    pos = torch.zeros(4, dtype=torch.int64, device=dev)
    slots = torch.arange(4, dtype=torch.int64, device=dev)
    out = ctypes.c_uint32(0)
    st = rq.lib().rq_validate_indices_noalloc(pos.data_ptr(), slots.data_ptr(), 4, 16,
                                              (1 << 20) + 1, ctypes.addressof(out),
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 2  # RQ_ERR_SHAPE
    assert _noalloc(pos, slots, 16, 1 << 20) == 0       # the largest size it takes
