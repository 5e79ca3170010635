"""Index bookkeeping of a ragged verify batch (requests with different numbers of draft tokens).

Source: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
"SpecDecodeMetadata: Index Bookkeeping".  The requests' scheduled tokens are laid end to end
(cu_num_scheduled_tokens is the running end of each request); a request with d draft tokens
needs the target's logits at its last d + 1 scheduled positions: d of them verify the drafts
and the last gives the bonus token.

Reading taken: the logits rows are those positions in request order, so request r's rows start
at (cu_num_draft_tokens[r] - d_r) + r; its first d_r rows are its draft-verification rows and
its last row is its bonus row.

Pinned by the worked example the page prints (tests/golden/spec_decode_metadata_5req.txt).

Paged cache addressing, from "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework",
section "EagleProposer: Draft Model Management": position pos of a sequence lives in slot
block_table[pos // block_size] * block_size + pos % block_size of the cache pool.  Pinned by its
invariants (tests/test_oracle_basics.py): every position of a sequence lands in one of its own
pages, consecutive positions of a page are consecutive slots, distinct positions of all
sequences with disjoint pages never share a slot, and a pool written position by position and
read back through the table is the contiguous cache.
"""
import numpy as np


def spec_decode_metadata(cu_num_scheduled_tokens, num_draft_tokens):
    """Returns a dict of int64 arrays: cu_num_draft_tokens, logits_indices (positions in the flat
    scheduled tokens), target_logits_indices and bonus_logits_indices (rows of the logits)."""
    cu = np.asarray(cu_num_scheduled_tokens, dtype=np.int64)
    d = np.asarray(num_draft_tokens, dtype=np.int64)
    if cu.shape != d.shape or (d < 0).any():
        raise ValueError("one non-negative draft count per request")
    starts = np.concatenate([[0], cu[:-1]])
    if (cu - starts < d + 1).any():
        raise ValueError("a request schedules fewer tokens than its drafts plus one")
    logits, target, bonus = [], [], []
    for r in range(len(cu)):
        first_row = len(logits)
        logits.extend(range(int(cu[r] - d[r] - 1), int(cu[r])))
        target.extend(range(first_row, first_row + int(d[r])))
        bonus.append(first_row + int(d[r]))
    return {"cu_num_draft_tokens": np.cumsum(d), "logits_indices": np.asarray(logits, np.int64),
            "target_logits_indices": np.asarray(target, np.int64),
            "bonus_logits_indices": np.asarray(bonus, np.int64)}


def slot_mapping(block_table_row, block_size, positions):
    """Pool slots of the given positions of one sequence (int64 array)."""
    bt = np.asarray(block_table_row, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    return bt[pos // block_size] * block_size + pos % block_size


def paged_view(pool, block_table_row, block_size, length):
    """The sequence's cache [length, ...] read from a pool [n_slots, ...] through its block table."""
    return np.asarray(pool)[slot_mapping(block_table_row, block_size, np.arange(length))]
