"""The collectives of ZeRO++ across real ranks, around the hot-path kernels.

On one GPU the library runs every virtual rank's buffers side by side and each exchange
is an index map inside the next kernel. Across real ranks (one process per GPU, launched
by torchrun) the exchanges are collectives, and this module runs them with
torch.distributed; the arithmetic between them stays in the library's kernels (the
`*_local` calls, which take one rank's own buffers).

Topology {N nodes, M GPUs per node}, W = N*M ranks, rank r = n*M + l. A gradient bucket
holds E elements per rank, cut into W slices of S = E/W; the hop-1 chunk is C = N*S.

* qwZ ("ZeRO++: Extremely Efficient Collective Communication for Large Model Training",
  atlas.scime.ai summary, Approach; the mlsanity.com record's Abstract): each rank
  quantises its block-aligned weight shard, the INT8 codes and fp32 scales are all-gathered
  (rank order = the flat weight order), and the gathered codes are dequantised.
* hpZ (same summary, Approach and Limitations): after the forward gather every rank keeps
  the slice l of the full fp16 weights (its node's secondary partition), so the backward
  gather runs inside the node only.
* qgZ (same summary, Approach; "LIT-102: ZeRO++ ..." Key takeaways): step 1 reorders and
  quantises the rank's bucket; hop 1 is an all-to-all inside the node (chunk l' goes to
  local peer l', chunk l of every peer comes back, peers in local-index order); the fused
  kernel reduces the M received chunks and requantises; hop 2 is an all-to-all across the
  nodes of the same local index (slice n' goes to node n', slice n of every node comes
  back, nodes in ascending order); the final kernel reduces the N received slices into the
  rank's owner slice.

The received buffers are bit for bit the slices of the single-GPU virtual layout that the
fused and final kernels read there (tested with the CPU oracle on gloo ranks), so the
result of every rank equals its row of the single-GPU exchange.
"""
import torch
import torch.distributed as dist

from . import binding as _b


class Groups:
    """The process groups of a topology. Every rank must construct it (collectively): each
    node's intra-node group and each local index's inter-node group are created on all
    ranks in the same order. Group ranks follow local index (node group) and node index
    (cross group), so an all-to-all over them runs in exactly the order the hops sum."""

    def __init__(self, N, M, rank=None):
        if not dist.is_initialized():
            raise RuntimeError("torch.distributed is not initialised")
        if dist.get_world_size() != N * M:
            raise ValueError(f"world size {dist.get_world_size()} != N*M = {N * M}")
        self.N, self.M, self.W = N, M, N * M
        self.rank = dist.get_rank() if rank is None else rank
        self.n, self.l = divmod(self.rank, M)
        self.node = self.cross = None
        for n in range(N):
            g = dist.new_group([n * M + l for l in range(M)])
            if n == self.n:
                self.node = g
        for l in range(M):
            g = dist.new_group([n * M + l for n in range(N)])
            if l == self.l:
                self.cross = g


# ----------------------------------------------------------------------------- qwZ / hpZ
def qwz_all_gather(codes, scales, group=None):
    """This rank's quantised shard (codes, scales) -> every rank's, concatenated in rank
    order: for block-aligned shards, the codes and scales of the whole flat weight set."""
    world = dist.get_world_size(group)
    gc = torch.empty(world * codes.numel(), dtype=codes.dtype, device=codes.device)
    gs = torch.empty(world * scales.numel(), dtype=scales.dtype, device=scales.device)
    dist.all_gather_into_tensor(gc, codes.reshape(-1), group=group)
    dist.all_gather_into_tensor(gs, scales.reshape(-1), group=group)
    return gc, gs


def hpz_secondary(full, groups):
    """This rank's part of its node's secondary partition: slice l of the full weights
    (M equal slices), kept after the forward gather."""
    if full.numel() % groups.M:
        raise ValueError("the weights do not split into M equal slices")
    per = full.numel() // groups.M
    return full.reshape(-1)[groups.l * per:(groups.l + 1) * per].clone()


def hpz_all_gather(secondary, groups):
    """The backward gather of hpZ: the node's M secondary slices -> the full weights, over
    the intra-node group only."""
    full = torch.empty(groups.M * secondary.numel(), dtype=secondary.dtype,
                       device=secondary.device)
    dist.all_gather_into_tensor(full, secondary.reshape(-1), group=groups.node)
    return full


# ----------------------------------------------------------------------------- qgZ hops
def _a2a(out, inp, group):
    dist.all_to_all_single(out.reshape(-1), inp.reshape(-1), group=group)
    return out


def hop1_all_to_all(codes, scales, groups, recv_codes=None, recv_scales=None):
    """Step-1 output of this rank (M chunks) -> chunk l of each rank of the node,
    [M][chunk] in local-index order (one all-to-all each for codes and scales)."""
    M = groups.M
    if recv_codes is None:
        recv_codes = torch.empty((M, codes.numel() // M), dtype=codes.dtype, device=codes.device)
    if recv_scales is None:
        recv_scales = torch.empty((M, scales.numel() // M), dtype=scales.dtype,
                                  device=scales.device)
    return _a2a(recv_codes, codes, groups.node), _a2a(recv_scales, scales, groups.node)


def hop1_p2p(codes, scales, groups, produce_chunk=None, recv_codes=None, recv_scales=None):
    """Hop 1 as point-to-point transfers in ring order: at step d the rank sends chunk
    (l + d) % M to that peer and receives from peer (l - d) % M. If `produce_chunk(p)` is
    given it is called just before chunk p is sent (it fills chunk p of codes / scales), so
    the quantisation of the next chunk overlaps the transfer of this one. The result equals
    hop1_all_to_all's."""
    M, l = groups.M, groups.l
    cb, sb = codes.numel() // M, scales.numel() // M
    if recv_codes is None:
        recv_codes = torch.empty((M, cb), dtype=codes.dtype, device=codes.device)
    if recv_scales is None:
        recv_scales = torch.empty((M, sb), dtype=scales.dtype, device=scales.device)
    node = [groups.n * M + j for j in range(M)]  # global ranks of the node's peers
    works = []
    for d in range(M):
        p, q = (l + d) % M, (l - d) % M
        if produce_chunk is not None:
            produce_chunk(p)
        cp, sp = codes.reshape(-1)[p * cb:(p + 1) * cb], scales.reshape(-1)[p * sb:(p + 1) * sb]
        if d == 0:  # this rank's own chunk stays
            recv_codes[l].copy_(cp)
            recv_scales[l].copy_(sp)
            continue
        ops = [dist.P2POp(dist.isend, cp, node[p], groups.node),
               dist.P2POp(dist.isend, sp, node[p], groups.node),
               dist.P2POp(dist.irecv, recv_codes[q], node[q], groups.node),
               dist.P2POp(dist.irecv, recv_scales[q], node[q], groups.node)]
        works += dist.batch_isend_irecv(ops)
    for w in works:
        w.wait()
    return recv_codes, recv_scales


def hop2_all_to_all(codes, scales, groups, recv_codes=None, recv_scales=None):
    """Hop-1 output of this rank (N slices) -> slice n of the hop-1 output of ranks
    (n', l), [N][slice] with n' ascending (one all-to-all each, inter-node group)."""
    N = groups.N
    if recv_codes is None:
        recv_codes = torch.empty((N, codes.numel() // N), dtype=codes.dtype, device=codes.device)
    if recv_scales is None:
        recv_scales = torch.empty((N, scales.numel() // N), dtype=scales.dtype,
                                  device=scales.device)
    return _a2a(recv_codes, codes, groups.cross), _a2a(recv_scales, scales, groups.cross)


# ----------------------------------------------------------------------------- one rank's step
def qgz_step(grads, block, bits, groups, post_scale=1.0, dtype=None, pipelined=False):
    """The whole qgZ exchange as this rank runs it on its GPU: step 1, hop 1, the fused
    hop, hop 2 and the final hop -> this rank's owner slice [E / W] (fp32 by default;
    post_scale 1/W averages). With `pipelined`, step 1 is run chunk by chunk and each
    chunk's transfer overlaps the quantisation of the next (hop1_p2p)."""
    N, M, W = groups.N, groups.M, groups.W
    E = grads.numel()
    C, S = E // M, E // W
    if pipelined:
        codes = torch.empty(_b.zpp_code_bytes(E, bits), dtype=torch.uint8, device=grads.device)
        scales = torch.empty(E // block, dtype=torch.float32, device=grads.device)

        def produce(p):
            _b.qgz_reorder_quant_local(grads, block, bits, N, M, codes, scales, chunks=(p, p + 1))

        rc, rs = hop1_p2p(codes, scales, groups, produce_chunk=produce)
    else:
        codes, scales = _b.qgz_reorder_quant_local(grads, block, bits, N, M)
        rc, rs = hop1_all_to_all(codes, scales, groups)
    c1, s1 = _b.dequant_reduce_requant_local(rc, rs, C, block, bits, M)
    r2c, r2s = hop2_all_to_all(c1, s1, groups)
    return _b.dequant_reduce_local(r2c, r2s, S, block, bits, N, post_scale=post_scale,
                                   dtype=dtype)
