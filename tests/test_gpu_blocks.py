"""The paged cache's block manager on the GPU against oracle.blocks.

A churn scenario runs kvc_block_prepare / kvc_block_share / kvc_block_release
and kvc_append on the device and the same steps on the oracle's
BlockManager, from the same free-list order.  After every call the device
state (block table, reference counts, free list and count, valid bits) must
equal the model's exactly; the cache must hold, at every attended position
of every sequence and layer, exactly the values that sequence appended (bf16,
no RoPE: bit-exact, copy-on-write copies included); decode outputs must
match the oracle's attention over each sequence's own history.
"""

import numpy as np
import pytest
import torch

from oracle import blocks as oblocks
from oracle.attention import decode_reference
from tests.gpu_harness import TOL

pytestmark = pytest.mark.gpu

L, B, HQ, HKV, D, BS, NB, MAXB = 2, 4, 8, 2, 128, 16, 24, 6


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_kvc_gb300 as m
    return m


class Scenario:
    def __init__(self, kvc, num_blocks=NB, seed=11, dtype="bf16"):
        self.kvc = kvc
        self.dtype = dtype
        self.d = kvc.make_desc("paged", "none", dtype, L, B, HQ, HKV, D, block_size=BS, num_blocks=num_blocks,
                               max_blocks_per_seq=MAXB)
        self.cache = kvc.alloc_cache(self.d, fill=0.0)
        self.ws = kvc.alloc_workspace(self.d)
        order = np.random.default_rng(seed).permutation(num_blocks).tolist()
        self.state = kvc.BlockState(self.d, free_order=order)
        self.bm = oblocks.BlockManager(num_blocks, BS, B, MAXB, free=order)
        self.hist = [dict() for _ in range(B)]        # b -> {pos: (k [L, HKV, D], v [L, HKV, D])}
        self.gen = torch.Generator().manual_seed(seed)

    def prepare_and_append(self, positions):
        pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
        self.kvc.block_prepare(self.d, self.cache, pos, self.state, self.ws)
        self.bm.prepare(positions)
        k = torch.randn((L, B, 1, HKV, D), generator=self.gen).to(torch.bfloat16)
        v = torch.randn((L, B, 1, HKV, D), generator=self.gen).to(torch.bfloat16)
        for layer in range(L):
            self.kvc.append(self.d, self.cache, layer, k[layer].cuda(), v[layer].cuda(), pos, self.ws,
                            block_table=self.state.table)
        for b, t in enumerate(positions):
            if t >= 0 and self.bm.table[b, t // BS] >= 0:
                self.hist[b][t] = (k[:, b, 0], v[:, b, 0])

    def share(self, src, dst, ntokens):
        nb = (ntokens + BS - 1) // BS
        t = lambda x: torch.tensor([x], dtype=torch.int32, device="cuda")
        self.kvc.block_share(self.d, self.state, t(src), t(dst), t(nb), self.ws)
        self.bm.share(src, dst, nb)
        self.hist[dst] = {p: kv for p, kv in self.hist[src].items() if p < ntokens}

    def release(self, seqs):
        self.kvc.block_release(self.d, self.state, torch.tensor(seqs, dtype=torch.int32, device="cuda"), self.ws)
        self.bm.release(seqs)
        for b in seqs:
            self.hist[b] = {}

    def check_state(self):
        torch.cuda.synchronize()
        st, bm = self.state, self.bm
        assert st.table.cpu().numpy().tolist() == bm.table.tolist()
        assert st.refcount.cpu().numpy().tolist() == bm.ref.tolist()
        n = int(st.free_count.item())
        assert n == len(bm.free)
        assert st.free_list[:n].cpu().numpy().tolist() == bm.free
        bits = st.valid_bits.cpu().numpy().view(np.uint32)
        valid = [(int(bits[i >> 5]) >> (i & 31)) & 1 == 1 for i in range(bm.num_blocks)]
        assert valid == bm.valid.tolist()
        assert bm.check_invariants()

    def check_cache(self):
        if self.dtype == "i8":
            # INT8 rows: codes and scales equal the oracle's quantisation of what was appended
            from oracle.quant import quantize_rows
            codes, scales = (x.cpu() for x in self.kvc.int8_views(self.d, self.cache))
            for b in range(B):
                for p, (k, v) in self.hist[b].items():
                    phys = self.bm.table[b, p // BS]
                    assert phys >= 0
                    for kv, x in ((0, k), (1, v)):
                        cq, sq = quantize_rows(x.float().numpy())
                        assert np.array_equal(codes[:, kv, phys, :, p % BS].numpy(), cq), (b, p, kv)
                        assert np.array_equal(scales[:, kv, phys, :, p % BS].numpy(), sq), (b, p, kv)
            return
        c = self.cache.cpu()
        for b in range(B):
            for p, (k, v) in self.hist[b].items():
                phys = self.bm.table[b, p // BS]
                assert phys >= 0
                assert torch.equal(c[:, 0, phys, :, p % BS], k), (b, p)
                assert torch.equal(c[:, 1, phys, :, p % BS], v), (b, p)

    def check_decode(self, positions):
        pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
        q = torch.randn((B, HQ, D), generator=self.gen).to(torch.bfloat16)
        g = HQ // HKV
        for layer in range(L):
            out = self.kvc.decode_attention(self.d, self.cache, layer, q.cuda(), pos, self.ws,
                                            block_table=self.state.table, valid_bits=self.state.valid_bits)
            got = out.float().cpu().numpy()
            for b, t in enumerate(positions):
                if t < 0:
                    continue
                ps = sorted(p for p in self.hist[b] if p <= t)
                for h in range(HKV):
                    K = np.stack([self.hist[b][p][0][layer, h].double().numpy() for p in ps])
                    V = np.stack([self.hist[b][p][1][layer, h].double().numpy() for p in ps])
                    if self.dtype == "i8":
                        from oracle.quant import store_i8
                        K, V = store_i8(K), store_i8(V)
                    ref = decode_reference(q[b, h * g:(h + 1) * g].double().numpy(), K, V, ps, t, rope="none",
                                           storage=self.dtype)
                    assert np.abs(got[b, h * g:(h + 1) * g] - ref).max() <= TOL["bf16"], (layer, b, h)


@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_block_manager_churn_matches_the_model(kvc, dtype):
    # INT8: copy-on-write copies carry the rows' scales with their codes
    sc = Scenario(kvc, dtype=dtype)
    # sequences 0 and 3 write 21 and 6 tokens
    for t in range(21):
        sc.prepare_and_append([t, -1, -1, t if t < 6 else -1])
        sc.check_state()
    sc.check_cache()
    # 1 takes 0's 21-token prefix (2 blocks, the second partly filled), 2 its first 16
    sc.share(0, 1, 21)
    sc.share(0, 2, 16)
    sc.check_state()
    # all advance: 0 copies the shared partial block (served first), 1 keeps it,
    # 2 starts a new block, 3 writes in place
    sc.prepare_and_append([21, 21, 16, 6])
    sc.check_state()
    assert sc.bm.table[0, 1] != sc.bm.table[1, 1]
    for step in range(1, 14):
        sc.prepare_and_append([21 + step, 21 + step, 16 + step, 6 + step])
        sc.check_state()
    sc.check_cache()
    sc.check_decode([34, 34, 29, 19])
    sc.release([0, 2])
    sc.check_state()
    sc.check_cache()
    assert kvc.get_error(sc.ws) == 0


def test_block_manager_runs_out_of_blocks(kvc):
    sc = Scenario(kvc, num_blocks=3, seed=5)
    sc.prepare_and_append([0, 0, 0, -1])
    sc.check_state()
    sc.prepare_and_append([-1, -1, -1, 0])          # no block left for sequence 3
    sc.check_state()
    assert kvc.get_error(sc.ws) & kvc.KVC_DEV_NO_FREE_BLOCK
    assert sc.bm.errors == [(3, oblocks.ERR_NO_FREE)]
