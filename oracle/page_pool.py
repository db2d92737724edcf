"""Plain reference of the page pool and prefix cache -- TEST INFRASTRUCTURE.

Only the test suite may import this module.  It restates, step by step, the
KV cache explainer's PagedAttention section (a pool of fixed-size pages, a
free list from which allocation pops a page id and to which freeing pushes it
back, pages shared between requests) and its Prefix Cache section (each full
block hashed over its tokens together with its parent block's hash; a lookup
walks a prompt's blocks in order and stops at the first miss, so the reused
length is floored to whole blocks), plus the Workers AI post's page tags
(§3: a page's tag changes each time it is handed out again).

The block hash is 64-bit FNV-1a (Fowler-Noll-Vo, variant 1a: offset basis
0xcbf29ce484222325, prime 0x100000001b3, xor then multiply per byte) over the
parent hash (8 bytes, little endian) and the block's token ids (4 bytes each,
little endian); the first block's parent is 0.  Parity pins:
tests/test_oracle_page_pool.py.
"""
from __future__ import annotations

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
_MASK = (1 << 64) - 1


class NoPages(Exception):
    pass


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & _MASK
    return h


def block_hash(parent: int, tokens) -> int:
    data = int(parent).to_bytes(8, "little") + b"".join((int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


def chain_hashes(tokens, page_size: int):
    """Hash of every full block of a token stream, each chained to the one before."""
    out, h = [], 0
    for i in range(len(tokens) // page_size):
        h = block_hash(h, tokens[i * page_size:(i + 1) * page_size])
        out.append(h)
    return out


class PagePool:
    def __init__(self, num_pages: int, page_size: int):
        self.page_size = page_size
        self.free = list(range(num_pages - 1, -1, -1))  # a stack: pops 0, 1, 2, ...
        self.ref = [0] * num_pages
        self.tag = [0] * num_pages
        self.prefix = {}      # block hash -> page
        self.hash_of = {}     # page -> the block hash it is registered under

    def map_request(self, tokens, max_pages: int):
        P = self.page_size
        n_pages = -(-len(tokens) // P)
        if n_pages > max_pages:
            raise ValueError("row too short")
        hashes = chain_hashes(tokens, P)
        hits = 0
        while hits < len(hashes) and hashes[hits] in self.prefix:   # stop at the first miss
            hits += 1
        if n_pages - hits > len(self.free):
            raise NoPages
        row, tags = [], []
        for i in range(n_pages):
            if i < hits:
                page = self.prefix[hashes[i]]
                self.ref[page] += 1
            else:
                page = self.free.pop()
                self.ref[page] = 1
                self.tag[page] += 1
                if i < len(hashes):
                    self.prefix[hashes[i]] = page
                    self.hash_of[page] = hashes[i]
            row.append(page)
            tags.append(self.tag[page])
        row += [-1] * (max_pages - n_pages)
        tags += [0] * (max_pages - n_pages)
        return row, tags, hits * P

    def release(self, row, n_pages: int):
        # each listed entry is one reference: a page listed k times needs k
        listed = {}
        for page in row[:n_pages]:
            listed[page] = listed.get(page, 0) + 1
        for page, k in listed.items():
            if page < 0 or page >= len(self.ref) or self.ref[page] < k:
                raise ValueError("not a held page")
        for page in row[:n_pages]:
            self.ref[page] -= 1
            if self.ref[page] == 0:
                h = self.hash_of.pop(page, None)
                if h is not None and self.prefix.get(h) == page:
                    del self.prefix[h]
                self.free.append(page)
