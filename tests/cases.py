"""Small geometries shared by the CPU emulator tests and the GPU parity tests."""
import workloads as wl

CASES = {
    "tiny": lambda: wl.tiny(),
    "tp4_to_tp8": lambda: wl.custom("a", 1, num_layers=3, num_components=2, kv_heads=8,
                                    head_dim=16, elem_bytes=2, src_tp=4, dst_tp=8,
                                    src_block=16, dst_block=32, seq_lens=[300, 1, 33]),
    "tp4_to_tp2_16_64": lambda: wl.custom("b", 2, num_layers=2, num_components=2, kv_heads=8,
                                          head_dim=8, elem_bytes=2, src_tp=4, dst_tp=2,
                                          src_block=16, dst_block=64,
                                          seq_lens=[700 - 5, 700 - 63, 64, 65]),
    "mla_64_16": lambda: wl.custom("c", 3, num_layers=2, num_components=1, kv_heads=1,
                                   head_dim=576, elem_bytes=2, src_tp=1, dst_tp=1,
                                   src_block=64, dst_block=16, seq_lens=[129, 64, 1000]),
    "tp3_to_tp2_odd": lambda: wl.custom("d", 4, num_layers=2, num_components=2, kv_heads=6,
                                        head_dim=8, elem_bytes=4, src_tp=3, dst_tp=2,
                                        src_block=3, dst_block=5, seq_lens=[40, 0, 17, 1],
                                        shared_prefix=2),
    "tp2_to_tp3_u8": lambda: wl.custom("e", 5, num_layers=2, num_components=2, kv_heads=6,
                                       head_dim=48, elem_bytes=1, src_tp=2, dst_tp=3,
                                       src_block=1, dst_block=7, seq_lens=[50, 9]),
    "big_block_1_to_64": lambda: wl.custom("f", 6, num_layers=1, num_components=2, kv_heads=4,
                                           head_dim=64, elem_bytes=2, src_tp=1, dst_tp=4,
                                           src_block=1, dst_block=64, seq_lens=[1000, 63]),
    # 256-token decode blocks of 8 x 128 heads: 1 MB tiles, cut into <= 64 KB slices
    "huge_block_16_to_256": lambda: wl.custom("g", 7, num_layers=2, num_components=2,
                                              kv_heads=8, head_dim=128, elem_bytes=2,
                                              src_tp=2, dst_tp=1, src_block=16,
                                              dst_block=256, seq_lens=[600, 256, 1]),
}
