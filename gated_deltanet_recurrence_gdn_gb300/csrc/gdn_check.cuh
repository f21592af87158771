// gdn_check.cuh -- the debug bounds-check build (-DGDN_BOUNDS_CHECK).
//
// Under the flag, the tcgen05 and chunk-prep kernels check every shared-memory
// access they make through the helpers (row stores, bulk-copy destinations,
// mbarriers, MMA operand descriptors), every tensor-memory column they load,
// and the global indices of their loads and stores against the sizes of the
// arrays.  A failed check skips the access and records the source line of the
// first failure in a word of its translation unit; gdn_sync_check() folds the
// words of all translation units into GDN_ERR_BOUNDS and
// gdn_bounds_violation() returns the line.  Nothing traps or asserts: the
// context stays usable.  Without the flag every check is the constant true and
// compiles away.
//
// Misaligned or out-of-range bulk-copy inputs fail silently or fault
// ("Gated DeltaNet GPU并行实现", section 5.2, second pitfall), so this build is
// the tool for finding an index error without a memory checker.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

#ifdef GDN_BOUNDS_CHECK

namespace gdn {

// Registers a reader of one translation unit's violation word (gdn_api.cu);
// read_clear returns the recorded line (0: none) and clears it if asked.
void register_bounds_word(int (*read_clear)(bool clear));

namespace chk {
namespace {

__device__ int g_first_violation;   // this translation unit's: line of the first failure

int read_clear(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_first_violation, sizeof(int)) != cudaSuccess) return 0;
    if (clear && v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_first_violation, &zero, sizeof(int));
    }
    return v;
}

struct Registrar {
    Registrar() { register_bounds_word(&read_clear); }
};
Registrar g_registrar;

}  // namespace

extern __shared__ __align__(16) uint8_t gdn_chk_dyn_smem[];

__device__ __forceinline__ bool fail(int line) {
    atomicCAS(&g_first_violation, 0, line);
    return false;
}

__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// [addr, addr + bytes) inside this CTA's dynamic shared memory
__device__ __forceinline__ bool smem_ok(uint32_t addr, uint32_t bytes, int line) {
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(gdn_chk_dyn_smem));
    return (addr >= base && addr - base + bytes <= dyn_smem_bytes()) || fail(line);
}

// 0 <= i and i + n <= size
__device__ __forceinline__ bool idx_ok(long long i, long long n, long long size, int line) {
    return (i >= 0 && i + n <= size) || fail(line);
}

// lane < 128 and column + ncols <= 512
__device__ __forceinline__ bool tmem_ok(uint32_t taddr, uint32_t ncols, int line) {
    return ((taddr >> 16) < 128u && (taddr & 0xFFFFu) + ncols <= 512u) || fail(line);
}

}  // namespace chk
}  // namespace gdn

#define GDN_SMEM_OK(addr, bytes) ::gdn::chk::smem_ok((addr), (bytes), __LINE__)
#define GDN_IDX_OK(i, n, size) \
    ::gdn::chk::idx_ok((long long)(i), (long long)(n), (long long)(size), __LINE__)
#define GDN_TMEM_OK(taddr, ncols) ::gdn::chk::tmem_ok((taddr), (ncols), __LINE__)

#else

#define GDN_SMEM_OK(addr, bytes) true
#define GDN_IDX_OK(i, n, size) true
#define GDN_TMEM_OK(taddr, ncols) true

#endif
