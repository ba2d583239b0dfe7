"""Host logic of the layer step without a GPU: the shard-major block table that lets one
launch run every emulated shard over a shared cache."""
import torch

from mla_paged_decode_03_gb300.layer_step import shard_major_block_table


def test_rows_are_offset_into_each_shards_slice():
    bt = torch.tensor([[0, 4, 2], [1, 3, 9]], dtype=torch.int32)   # 9 is past every pool
    out = shard_major_block_table(bt, [5, 3, 4])
    assert out.shape == (6, 3) and out.dtype == torch.int32 and out.is_contiguous()
    # shard 0: ids < 5 kept, 9 out of range
    assert out[0].tolist() == [0, 4, 2]
    assert out[1].tolist() == [1, 3, -1]
    # shard 1 (3 blocks, offset 5): 4 and 3 are outside its pool
    assert out[2].tolist() == [5, -1, 7]
    assert out[3].tolist() == [6, -1, -1]
    # shard 2 (4 blocks, offset 8)
    assert out[4].tolist() == [8, -1, 10]
    assert out[5].tolist() == [9, 11, -1]


def test_negative_ids_stay_negative_and_one_shard_is_identity():
    bt = torch.tensor([[-1, 0, 2]], dtype=torch.int32)
    assert shard_major_block_table(bt, [3]).tolist() == [[-1, 0, 2]]
    two = shard_major_block_table(bt, [3, 3])
    assert two.tolist() == [[-1, 0, 2], [-1, 3, 5]]


def test_wide_strided_table_is_compacted():
    wide = torch.arange(10, dtype=torch.int32).view(2, 5)[:, :3]   # row stride 5
    out = shard_major_block_table(wide, [10, 10])
    assert out.stride(0) == 3
    assert out[2].tolist() == [10, 11, 12] and out[3].tolist() == [15, 16, 17]
