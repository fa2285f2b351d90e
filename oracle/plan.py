"""Split-KV partition rule for decode, restated plainly (test infrastructure).

The library's plan scheduler must produce exactly these int32 words.  The
rule (the pages only say that the plan splits KV across CTAs, with
fixed-split and disable-split options; the balanced rule is this library's):

* Rows are (request b, KV-head block hb), row r = b * nhb + hb, where a block
  holds hpc KV heads, hpc = the largest divisor of num_kv_heads that is <= 8,
  and nhb = num_kv_heads / hpc.  Row r holds npages[b] pages of 16 tokens:
  ceil(kv_len / 16), where kv_len = (pages - 1) * page_size + last_page_len
  (a page of page_size = 16 m tokens counts as m 16-token pages; for
  page_size 16 this is the request's page count).
* disable_split_kv: one segment (r, 0, npages) per non-empty row; segment k
  goes to CTA k mod G, G = min(num_ctas, #segments).
* fixed_split_pages = c > 0: each row cut into [0,c), [c,2c), ...; dealt the
  same way.
* otherwise (balanced): T = total pages of all rows, G = min(num_ctas, T).
  When T >= 16 G and 4 R >= G (R rows), the last npages // 16 pages of every
  row are handed out at run time (none otherwise); the rows' first ns pages
  (the rest) are laid end to end, Ts = sum ns, and CTA i owns static pages
  [i*Ts//G, (i+1)*Ts//G), cut at row boundaries.  The run-time pages of each
  row, [ns, npages), are cut into chunks of c = max(4, ceil(Td / G)) pages,
  Td = T - Ts (the last chunk of a row may be shorter); chunks are listed in
  row and page order after every CTA's segments and numbered with them.
* Rows with no pages get a zero-page segment (r, 0, 0); the k-th such row
  (ascending r) goes to CTA k mod G, after that CTA's other segments.  If no
  row has pages, G = 1 when some row exists.
* Within each CTA, segments that cover only part of their row come first
  (keeping their order), then the rest.
* A segment that spans its whole row (including a zero-page one) has
  out_slot -1; the others get slots 0, 1, 2, ... row by row (merge rows
  ascending), and within a row by first page, so each merge row's slots are
  consecutive.
* Merge rows: rows with two or more segments (chunks count as segments),
  ascending; each lists its slots ordered by first page (so the slot list is
  0, 1, 2, ...).  row_merge[r] is the merge entry of row r, or -1.  A
  separate merge pass combines each merge row's slots in that order.
* Header word 22 holds the number of chunks, word 23 the offset of their
  (row, first page, end page, slot) records.
"""
from __future__ import annotations

HEADER_WORDS = 32
MAGIC = 0x38464150
DYN_DIV, DYN_CHUNKS_PER_CTA, DYN_MIN_CHUNK, DYN_MIN_PAGES_PER_CTA, DYN_MIN_ROWS_DIV = 16, 1, 4, 16, 4


def heads_per_cta(num_kv_heads: int) -> int:
    return max(d for d in range(1, 9) if num_kv_heads % d == 0)


def decode_metadata(kv_indptr, last_page_len, *, num_qo_heads, num_kv_heads, num_ctas,
                    page_size=16, fixed_split_pages=0, disable_split_kv=False):
    kv_indptr = [int(x) for x in kv_indptr]
    last_page_len = [int(x) for x in last_page_len]
    B = len(kv_indptr) - 1
    hpc = heads_per_cta(num_kv_heads)
    nhb = num_kv_heads // hpc
    group = num_qo_heads // num_kv_heads
    npages = []
    for b in range(B):
        n = kv_indptr[b + 1] - kv_indptr[b]
        kv = (n - 1) * page_size + last_page_len[b] if n > 0 else 0
        for _ in range(nhb):
            npages.append((kv + 15) // 16)
    R = B * nhb

    per_cta = []
    chunks = []
    if disable_split_kv or fixed_split_pages > 0:
        segs = []
        for r in range(R):
            c = npages[r] if disable_split_kv else fixed_split_pages
            a = 0
            while a < npages[r]:
                segs.append([r, a, min(a + c, npages[r]), 0])
                a += c
        G = min(num_ctas, len(segs))
        per_cta = [[] for _ in range(G)]
        for k, s in enumerate(segs):
            per_cta[k % G].append(s)
    else:
        T = sum(npages)
        G = min(num_ctas, T)
        dyn = G > 0 and T >= DYN_MIN_PAGES_PER_CTA * G and R * DYN_MIN_ROWS_DIV >= G
        ns = [n - n // DYN_DIV if dyn else n for n in npages]
        Ts = sum(ns)
        Td = T - Ts
        per_cta = [[] for _ in range(G)]
        starts = [0]
        for n in ns:
            starts.append(starts[-1] + n)
        for i in range(G):
            lo, hi = i * Ts // G, (i + 1) * Ts // G
            for r in range(R):
                a = max(lo, starts[r]) - starts[r]
                e = min(hi, starts[r + 1]) - starts[r]
                if e > a:
                    per_cta[i].append([r, a, e, 0])
        if Td > 0:
            c = max(DYN_MIN_CHUNK, -(-Td // (DYN_CHUNKS_PER_CTA * G)))
            for r in range(R):
                for a in range(ns[r], npages[r], c):
                    chunks.append([r, a, min(a + c, npages[r]), 0])

    empty = [r for r in range(R) if npages[r] == 0]
    if empty and not per_cta:
        per_cta = [[]]
    for k, r in enumerate(empty):
        per_cta[k % len(per_cta)].append([r, 0, 0, 0])

    def is_partial(sg):
        return not (sg[1] == 0 and sg[2] == npages[sg[0]])

    per_cta = [[sg for sg in segs if is_partial(sg)] + [sg for sg in segs if not is_partial(sg)]
               for segs in per_cta]

    seg_count = [0] * R
    row_parts = [[] for _ in range(R)]
    for segs in per_cta + [chunks]:
        for s in segs:
            seg_count[s[0]] += 1
            if not is_partial(s):
                s[3] = -1
            else:
                row_parts[s[0]].append(s)
    slot = 0
    merge_rows, merge_ptr, merge_slots = [], [0], []
    row_merge = [-1] * R
    for r in range(R):
        if seg_count[r] >= 2:
            row_merge[r] = len(merge_rows)
            merge_rows.append(r)
            for s in sorted(row_parts[r], key=lambda sg: sg[1]):
                s[3] = slot
                merge_slots.append(slot)
                slot += 1
            merge_ptr.append(len(merge_slots))

    req_page = [kv_indptr[b] for b in range(B)]
    req_kv = []
    for b in range(B):
        n = kv_indptr[b + 1] - kv_indptr[b]
        req_kv.append((n - 1) * page_size + last_page_len[b] if n > 0 else 0)
    cta_ptr = [0]
    flat = []
    for segs in per_cta:
        cta_ptr.append(cta_ptr[-1] + len(segs))
        for s in segs:
            flat += s

    words = [0] * HEADER_WORDS
    words[0] = MAGIC
    words[1] = 0
    words[2] = B
    words[3] = nhb
    words[4] = hpc
    words[5] = group
    words[6] = len(per_cta)
    words[7] = sum(len(s) for s in per_cta)
    words[8] = slot
    words[9] = len(merge_rows)

    def put(field, arr):
        words[field] = len(words)
        words.extend(arr)

    put(10, req_page)
    put(11, req_kv)
    put(12, cta_ptr)
    put(13, flat)
    put(14, merge_ptr)
    put(15, merge_rows)
    put(16, merge_slots)
    put(21, row_merge)
    words[22] = len(chunks)
    put(23, [x for ch in chunks for x in ch])
    return words


def prefill_metadata(kv_indptr, last_page_len, qo_indptr, *, num_qo_heads, num_kv_heads, num_ctas,
                     page_size=16, head_dim=128, kv_dtype="e4m3fn"):
    """Prefill work items.  TQ = 128 // group new tokens fill a 128-row
    query tile.  With a 2-byte cache (f16, bf16) at head_dim 128 two CTAs
    work as a pair on each query tile of 2 * TQ tokens (TQ per CTA);
    otherwise one CTA works on a tile of TQ tokens.  For request b, KV head hk and each block of two such tiles
    (A, then B right after) starting at t0, one item; its KV-tile count is
    the number of 128-key tiles its last token may see under the
    bottom-right causal rule, capped by the request's own key tiles.
    Each tile record is (b, hk, t0, nkv, qo_indptr[b], qo_len, kv_len,
    kv_indptr[b]).  Tiles are sorted by that count, descending, ties in
    (b, hk, t0) order.  G = min(num_ctas, #items) persistent CTAs (pairs:
    G = 2 min(max(1, num_ctas // 2), #items) CTAs, G / 2 pairs) take the
    items in snake order: in round r worker i takes item r W + i for even r
    and r W + W - 1 - i for odd r (W = G, or G / 2 pairs).  The order is
    the kernels'; the metadata holds the list."""
    kv_indptr = [int(x) for x in kv_indptr]
    last_page_len = [int(x) for x in last_page_len]
    qo_indptr = [int(x) for x in qo_indptr]
    B = len(kv_indptr) - 1
    group = num_qo_heads // num_kv_heads
    TQ = 128 // group
    pair = head_dim == 128 and kv_dtype in ("f16", "bf16")
    span = (4 if pair else 2) * TQ  # tokens per item
    req_page, req_kv, tiles = [], [], []
    for b in range(B):
        n = kv_indptr[b + 1] - kv_indptr[b]
        kv = (n - 1) * page_size + last_page_len[b] if n > 0 else 0
        req_page.append(kv_indptr[b])
        req_kv.append(kv)
        qo = qo_indptr[b + 1] - qo_indptr[b]
        for hk in range(num_kv_heads):
            for t0 in range(0, qo, span):
                last = min(t0 + span, qo) - 1
                lim = last + kv - qo
                nkv = min((kv + 127) // 128, lim // 128 + 1)
                tiles.append((b, hk, t0, nkv, qo_indptr[b], qo, kv, kv_indptr[b]))
    tiles = sorted(tiles, key=lambda t: -t[3])  # stable
    G = 2 * min(max(1, num_ctas // 2), len(tiles)) if pair else min(num_ctas, len(tiles))
    words = [0] * HEADER_WORDS
    words[0] = MAGIC
    words[1] = 1
    words[2] = B
    words[3] = num_kv_heads
    words[4] = 1
    words[5] = group
    words[6] = G
    words[18] = len(tiles)
    words[20] = TQ

    def put(field, arr):
        words[field] = len(words)
        words.extend(arr)

    put(10, req_page)
    put(11, req_kv)
    put(17, qo_indptr)
    put(19, [x for t in tiles for x in t])
    return words
