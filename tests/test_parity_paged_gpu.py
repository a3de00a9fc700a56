"""Prefill and decode over a paged key/value cache against the CPU oracle on
the same keys laid out contiguously, through the C ABI.  Pages are handed out
in a seeded random order; pages no sequence owns are filled with NaN, so a
read of a wrong page shows up in the outputs."""
import numpy as np
import pytest

import inputgen
import oracle
import parity

pytestmark = pytest.mark.gpu
NAN_BF16 = 0x7FC0
STREAM_PAGES = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import gqa_attention_prefill_gb300 as pkg
    from gqa_attention_prefill_gb300 import build
    build.build()
    pkg.load_library()


def paginate(w, page_size, extra_pages=5):
    """(k_pool, v_pool, block_table, num_pages, max_blocks) for workload w."""
    lens = [int(x) for x in w.seqlens_k]
    nb = [(L + page_size - 1) // page_size for L in lens]
    num_pages = sum(nb) + extra_pages
    max_blocks = max(nb) + 2
    order = np.argsort(inputgen.uniform_int(w.seed, STREAM_PAGES, num_pages, 0, 1 << 30),
                       kind="stable")
    shape = (num_pages, page_size, w.Hkv, w.D)
    kp = np.full(shape, NAN_BF16, dtype=np.uint16)
    vp = np.full(shape, NAN_BF16, dtype=np.uint16)
    table = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    fill = inputgen.normal_bf16(w.seed, STREAM_PAGES + 1, (page_size, w.Hkv, w.D))
    nxt = 0
    for s, L in enumerate(lens):
        k0 = int(w.cu_seqlens_k[s])
        for b in range(nb[s]):
            pg = int(order[nxt]); nxt += 1
            table[s, b] = pg
            n = min(page_size, L - b * page_size)
            kp[pg] = fill  # finite values in the slots past the sequence's end
            vp[pg] = fill
            kp[pg, :n] = w.k[k0 + b * page_size:k0 + b * page_size + n]
            vp[pg, :n] = w.v[k0 + b * page_size:k0 + b * page_size + n]
    return kp, vp, table, num_pages, max_blocks


def run_paged(w, page_size, decode=False, table_edit=None, check_status=True):
    import torch
    import gqa_attention_prefill_gb300 as pkg
    kp, vp, table, num_pages, max_blocks = paginate(w, page_size)
    if table_edit:
        table_edit(table)
    dev = "cuda"
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    q = to(w.q)
    k_pool, v_pool = to(kp), to(vp)
    tab = torch.from_numpy(table).to(dev)
    cu_q = torch.from_numpy(w.cu_seqlens).to(dev)
    cu_k = torch.from_numpy(w.cu_seqlens_k).to(dev)
    sinks = None if w.sinks is None else torch.from_numpy(w.sinks).to(dev)
    T = w.total_tokens
    out = torch.full((T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((T, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    if decode:
        rc = pkg.tsk_mha_decode_paged(q, k_pool, v_pool, sinks, cu_k, tab, max_blocks, page_size,
                                      num_pages, w.num_seqs, w.total_keys, max(w.seqlens_k),
                                      w.Hq, w.Hkv, w.D, w.window, w.scale, out, lse)
    else:
        rc = pkg.tsk_mha_prefill_paged(q, k_pool, v_pool, sinks, cu_q, cu_k, tab, max_blocks,
                                       page_size, num_pages, w.num_seqs, T, w.total_keys, w.Hq,
                                       w.Hkv, w.D, w.window, w.scale, out, lse)
    assert rc == 0, f"{pkg.STATUS.get(rc, rc)} {pkg.tsk_last_error()}"
    torch.cuda.synchronize()
    st = pkg.tsk_get_device_status()
    if check_status:
        assert st == 0, pkg.STATUS.get(st, st)
    return out, lse, st


def check(w, page_size, decode=False, label=""):
    out, lse, _ = run_paged(w, page_size, decode)
    ro, rl, _ = oracle.run_workload(w)
    return parity.compare(out.float().cpu().numpy().astype(np.float64),
                          lse.cpu().numpy().astype(np.float64), ro, rl, label)


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
def test_prefill_page_sizes(page_size):
    w = inputgen.make_kvcache([1, 100, 300, 129], [50, 1000, 300, 2049], 8, 2, seed=page_size)
    print(check(w, page_size, label=f"prefill page={page_size}"))


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_decode_page_sizes(page_size):
    w = inputgen.make_kvcache([1] * 5, [1, 17, 1000, 5000, 129], 16, 2, seed=page_size + 1)
    print(check(w, page_size, decode=True, label=f"decode page={page_size}"))


@pytest.mark.parametrize("decode", [False, True])
@pytest.mark.parametrize("window", [5, 128, 300])
def test_windows(decode, window):
    q = [1] * 3 if decode else [7, 200, 1]
    w = inputgen.make_kvcache(q, [900, 257, 3000], 8, 2, window=window, seed=window)
    print(check(w, 32, decode=decode, label=f"{'decode' if decode else 'prefill'} W={window}"))


@pytest.mark.parametrize("decode", [False, True])
def test_head_dim_128(decode):
    q = [1] * 3 if decode else [64, 300, 1]
    w = inputgen.make_kvcache(q, [700, 300, 2500], 32, 8, D=128, scale=128 ** -0.5, seed=9)
    print(check(w, 64, decode=decode, label=f"D=128 {'decode' if decode else 'prefill'}"))


@pytest.mark.parametrize("decode", [False, True])
def test_bad_page_index_reported(decode):
    import torch
    q = [1, 1] if decode else [10, 20]
    w = inputgen.make_kvcache(q, [300, 500], 8, 2, seed=4)

    def corrupt(table):
        table[1, 1] = 10 ** 6  # beyond the pool
    out, lse, st = run_paged(w, 64, decode=decode, table_edit=corrupt, check_status=False)
    assert st == -8
    assert torch.isnan(out.float()).all()


@pytest.mark.parametrize("page_size", [16, 128])
@pytest.mark.parametrize("window", [0, 200])
def test_prefill_one_query_head_per_kv_head(page_size, window):
    # Hq == Hkv: a work unit is two consecutive 128-row tiles of one head, the
    # second tile's keys read through the block table too; an odd number of
    # query tiles in the second sequence, sequence ends inside either tile
    w = inputgen.make_kvcache([129, 300], [700, 2500], 4, 4, window=window,
                              seed=page_size + window)
    print(check(w, page_size, label=f"prefill G=1 page={page_size} W={window}"))
