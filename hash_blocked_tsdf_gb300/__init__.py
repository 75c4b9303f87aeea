"""Hash-blocked TSDF integration (allocate + update) for one NVIDIA GB300.

The compute path lives in ``libtsdf.so`` (CUDA, sm_103a) behind the C ABI of
``include/tsdf.h``; ``binding`` marshals PyTorch tensors into it.
``scenes`` synthesises seeded input frames.
"""
from .binding import (TsdfError, TsdfVolume, load_library, tsdf_allocate, tsdf_allocate_batch,
                      tsdf_allocate_blocks, tsdf_update_batch,
                      tsdf_block_count, tsdf_clear_stats, tsdf_create, tsdf_destroy,
                      tsdf_export_blocks, tsdf_export_table, tsdf_extract_triangles,
                      tsdf_import_blocks, tsdf_get_info, tsdf_get_pool, tsdf_get_stats,
                      tsdf_integrate, tsdf_integrate_batch, tsdf_integrate_batch_host,
                      tsdf_reset, tsdf_set_instrumentation, tsdf_set_occlusion,
                      tsdf_set_pool_layout, tsdf_set_update_kernel, tsdf_update)

__all__ = [
    "TsdfError", "TsdfVolume", "load_library", "tsdf_allocate", "tsdf_allocate_batch",
    "tsdf_allocate_blocks", "tsdf_update_batch",
    "tsdf_block_count", "tsdf_clear_stats", "tsdf_create", "tsdf_destroy", "tsdf_export_blocks",
    "tsdf_export_table", "tsdf_extract_triangles", "tsdf_import_blocks", "tsdf_get_info", "tsdf_get_pool", "tsdf_get_stats", "tsdf_integrate",
    "tsdf_integrate_batch", "tsdf_integrate_batch_host", "tsdf_reset",
    "tsdf_set_instrumentation", "tsdf_set_occlusion", "tsdf_set_pool_layout",
    "tsdf_set_update_kernel", "tsdf_update",
]
