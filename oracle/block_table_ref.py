"""CPU oracle for building the decode's block table from a request pool.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this file: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  It shares no code, table or helper with the CUDA path.

The serving pages build the per-request page list the decode reads in one of
two ways, both written out here as plain loops, one entry at a time:

* From a token pool (sglang ``trtllm_mla_backend.py``,
  ``TRTLLMMLABackend._create_block_kv_indices`` and the graph-replay body
  that calls ``create_flashmla_kv_indices_triton``): ``req_to_token[r, j]``
  is the cache slot of token j of pool row r, and the table is first filled
  with -1.  The pages show only the kernel's arguments (pool, row indices,
  lengths, page size, max_blocks).  Reading taken: the cache is viewed as
  ``[num_pages, page_size, 576]`` (``forward_decode``), so slot t lives in
  page ``t // page_size``; entry i < ceil(L / page_size) of request b is the
  page of the first token of its page i, ``req_to_token[pool[b], i * page]
  // page``, and every other entry stays -1.
* From a page pool (tokenspeed ``trtllm_mla.py``,
  ``TRTLLMMLABackend._create_block_kv_indices``; tokenspeed ``flashmla.py``,
  ``_init_decode_metadata``): a gather of the first ``min(max_blocks,
  pool columns)`` columns of ``req_to_page[pool[b]]``; the table starts as
  zeros, so entries past those columns are 0.

parity pinned: tests/test_block_table_oracle.py checks both against tables
written out by hand and against each other on pools built from a known page
list.
"""

from __future__ import annotations

import numpy as np


def block_table_from_tokens(req_to_token: np.ndarray, req_pool_indices: np.ndarray, seq_lens: np.ndarray,
                            page_size: int, max_blocks: int) -> np.ndarray:
    """int32 [batch, max_blocks]: page ids of each request's pages, -1 after
    ceil(seq_len / page_size) entries (the token-pool construction)."""
    req_to_token = np.asarray(req_to_token)
    batch = len(req_pool_indices)
    table = np.full((batch, max_blocks), -1, dtype=np.int64)
    for b in range(batch):
        row = int(req_pool_indices[b])
        length = int(seq_lens[b])
        pages = (length + page_size - 1) // page_size
        for i in range(min(pages, max_blocks)):
            first_token_slot = int(req_to_token[row, i * page_size])
            table[b, i] = first_token_slot // page_size
    return table.astype(np.int32)


def block_table_from_pages(req_to_page: np.ndarray, req_pool_indices: np.ndarray,
                           max_blocks: int) -> np.ndarray:
    """int32 [batch, max_blocks]: the first min(max_blocks, pool columns)
    entries of each request's pool row, 0 after them (the page-pool
    construction)."""
    req_to_page = np.asarray(req_to_page)
    batch = len(req_pool_indices)
    copy_len = min(max_blocks, req_to_page.shape[1])
    table = np.zeros((batch, max_blocks), dtype=np.int64)
    for b in range(batch):
        row = int(req_pool_indices[b])
        for i in range(copy_len):
            table[b, i] = int(req_to_page[row, i])
    return table.astype(np.int32)
