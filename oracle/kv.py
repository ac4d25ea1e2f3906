"""Oracle: where request b's key s lives in a KV buffer.

Test infrastructure only (see the package docstring).

Contiguous: the KV of the whole batch is in logical (flattened) order after the rerange, so
request b's key s is row cu[b] + s ("[DeepSeek v3.2] 上下文并行详解", section 4 part 3 step B).
Paged: a decode-style cache of fixed-size pages; key s of request b is row
block_table[b, s // page] * page + s % page.
"""
from __future__ import annotations

import numpy as np


class ContiguousKV:
    def __init__(self, cu):
        self.cu = np.asarray(cu, dtype=np.int64)

    def rows(self, b: int, s: np.ndarray) -> np.ndarray:
        return self.cu[b] + np.asarray(s, dtype=np.int64)


class PagedKV:
    def __init__(self, block_table, page_size: int):
        self.table = np.asarray(block_table, dtype=np.int64)
        self.page = int(page_size)

    def rows(self, b: int, s: np.ndarray) -> np.ndarray:
        s = np.asarray(s, dtype=np.int64)
        return self.table[b, s // self.page] * self.page + s % self.page
