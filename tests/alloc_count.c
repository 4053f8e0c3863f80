/*
 * Host-allocation counter for the decode-step tests (test infrastructure).
 *
 * Preloaded (LD_PRELOAD) into a child process, it interposes the C library's
 * allocation entry points -- malloc, calloc, realloc, memalign,
 * posix_memalign, aligned_alloc; C++ operator new calls malloc -- counts each
 * call on the calling thread, and forwards it to the C library's own
 * implementation.  qg_test_thread_allocs() returns the calling thread's count,
 * so a test can bracket a call of the library and see how many host
 * allocations it made on that thread, through every layer below it (the
 * library, the C++ runtime, the CUDA runtime and driver).  This is the
 * counting allocator of aprender PR #4332 ("Greedy GPU argmax", counters
 * table: host allocations per token), done at the C library's boundary.
 */
#include <stddef.h>

extern void* __libc_malloc(size_t n);
extern void* __libc_calloc(size_t a, size_t b);
extern void* __libc_realloc(void* p, size_t n);
extern void* __libc_memalign(size_t align, size_t n);
extern void __libc_free(void* p);

/* initial-exec TLS: reading it never calls into the allocator */
static __thread unsigned long long n_alloc __attribute__((tls_model("initial-exec")));

unsigned long long qg_test_thread_allocs(void) { return n_alloc; }

void* malloc(size_t n) {
    ++n_alloc;
    return __libc_malloc(n);
}
void* calloc(size_t a, size_t b) {
    ++n_alloc;
    return __libc_calloc(a, b);
}
void* realloc(void* p, size_t n) {
    ++n_alloc;
    return __libc_realloc(p, n);
}
void free(void* p) { __libc_free(p); }
void* memalign(size_t align, size_t n) {
    ++n_alloc;
    return __libc_memalign(align, n);
}
void* aligned_alloc(size_t align, size_t n) {
    ++n_alloc;
    return __libc_memalign(align, n);
}
int posix_memalign(void** out, size_t align, size_t n) {
    ++n_alloc;
    void* p = __libc_memalign(align, n);
    if (!p) return 12; /* ENOMEM */
    *out = p;
    return 0;
}
